"""GB300-native route-set sparse GQA attention (QSA).

Exact grouped-query attention in which every query row attends only to its own
list of K/V token IDs, as the NeMo-AutoModel Qwen3.8-Flash-Next pages define it
(flex_qsa, fa4_qsa, qsa).  The work runs in libqsa, a C-ABI library of CUDA
kernels for sm_103a (``include/qsa.h``); this package is its PyTorch binding.
The same library produces the routes (``include/qsa_route.h``,
:func:`select_qsa_token_ids`: compressed-block scores and top-k selection).

Importing the package does not load the library; the first call does, and
raises if it has not been built (``route_sparse_gqa_gb300.build.build()``).
"""
from ._abi import EXPORTS, QSAError
from .attention import (RoutePlan, backward, forward, preprocess, qsa_attention, qsa_attention_with_lse,
                        resolve_scale)
from .routes import index_scores, select_from_scores, select_qsa_token_ids

__all__ = [
    "EXPORTS",
    "QSAError",
    "RoutePlan",
    "backward",
    "forward",
    "index_scores",
    "preprocess",
    "qsa_attention",
    "qsa_attention_with_lse",
    "resolve_scale",
    "select_from_scores",
    "select_qsa_token_ids",
]
