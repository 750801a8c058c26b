"""DeepSeek Sparse Attention (DSA) forward path for one GB300 GPU.

The compute path is libdsa.so (hand-written CUDA for sm_103a, C ABI in
include/dsa.h): lightning indexer -> exact top-k -> sparse MLA in MQA mode,
with IndexShare reuse of one index set across a group of layers, and an
HBM least-recently-used cache of latent rows over pinned host memory.
"""
from . import _lib
from .api import HiSparseCache, SparseAttention, SparseMHA

__all__ = ["SparseAttention", "SparseMHA", "HiSparseCache", "_lib"]
