"""GB300-native attention over a paged KV cache.

libwf.so (CUDA kernels for sm_103a behind the C ABI in include/wf.h) does the
work; ``binding`` marshals torch tensors to it; ``workloads`` draws seeded
synthetic inputs; ``build`` compiles the library in-tree.

Importing the package loads nothing: the library is loaded on the first call
and a missing library raises (there is no fallback path).
"""
__all__ = ["binding", "workloads", "build"]
