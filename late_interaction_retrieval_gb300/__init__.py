"""GB300-native late-interaction MaxSim.

The operator (Late Interaction Kernels README, "What does it compute?"):
score(q, d) = sum over valid query tokens i of max over valid document
tokens j of Q_i . D_j, in three layouts (all-pairs, pairwise, per-query
candidates) with a backward for each.  All arithmetic runs in the CUDA
library ``liblik`` (C ABI in ``include/lik.h``); this package only builds it,
loads it and marshals torch tensors into its calls.

``workloads`` (seeded synthetic inputs) imports without the CUDA library.
The binding and the autograd layers load it on first use and fail loudly
when it is missing.
"""
import importlib

__all__ = ["binding", "layers", "workloads", "MaxSim", "MaxSimPairwise", "MaxSimKD",
           "maxsim", "maxsim_pairwise", "maxsim_kd", "LIKError"]

_LAZY = {
    "binding": ("late_interaction_retrieval_gb300.binding", None),
    "layers": ("late_interaction_retrieval_gb300.layers", None),
    "MaxSim": ("late_interaction_retrieval_gb300.layers", "MaxSim"),
    "MaxSimPairwise": ("late_interaction_retrieval_gb300.layers", "MaxSimPairwise"),
    "MaxSimKD": ("late_interaction_retrieval_gb300.layers", "MaxSimKD"),
    "maxsim": ("late_interaction_retrieval_gb300.layers", "maxsim"),
    "maxsim_pairwise": ("late_interaction_retrieval_gb300.layers", "maxsim_pairwise"),
    "maxsim_kd": ("late_interaction_retrieval_gb300.layers", "maxsim_kd"),
    "LIKError": ("late_interaction_retrieval_gb300.binding", "LIKError"),
}


def __getattr__(name):
    if name == "workloads":
        return importlib.import_module("late_interaction_retrieval_gb300.workloads")
    if name not in _LAZY:
        raise AttributeError(name)
    mod, attr = _LAZY[name]
    m = importlib.import_module(mod)
    return m if attr is None else getattr(m, attr)
