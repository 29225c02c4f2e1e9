"""Scaled dot-product attention forward for NVIDIA GB300 (sm_103a).

The compute lives in libsdpa.so (C ABI in include/sdpa.h); ``sdpa`` is its Python binding,
``contracts`` maps the ai.onnx Attention, MultiHeadAttention and GroupQueryAttention
operator contracts onto it, and ``workloads`` draws seeded synthetic inputs.
Importing the package loads nothing; the library is loaded on first use.
"""
__all__ = ["sdpa", "workloads"]
