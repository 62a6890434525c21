"""Batch-invariant bf16 linear layer for GB300 (sm_103a).

The compute runs in the CUDA library ``libbi_gemm.so`` built from ``csrc/``;
``binding`` marshals torch tensors into its C ABI (declared in
``include/bi_gemm.h``).  Nothing is imported eagerly, so ``inputs`` can be used
on a machine where the library is not built.
"""

__all__ = ["binding", "inputs", "build"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(__name__ + "." + name)
    raise AttributeError(name)
