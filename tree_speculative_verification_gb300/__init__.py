"""GB300 (sm_103a) tree-based speculative verification.

The hot path of one verification step of SpecInfer-style tree speculative
inference (arXiv 2305.09781): depth-first tree linearisation, shared tree KV
cache append/commit, split-KV tree attention with a topology-aware mask, and
greedy / multi-step-speculative-sampling verification, all as CUDA kernels
behind the C ABI of include/treespec.h. ``api`` is the thin Python binding.
"""
from . import workloads  # noqa: F401

__all__ = ["api", "workloads", "step", "build"]
