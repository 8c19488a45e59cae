"""GB300-native MXFP4 mixture-of-experts FFN layer (softmax top-K routing).

The compute lives in the C-ABI CUDA library ``libmoe`` (csrc/, declared in
include/moe.h); the submodule ``libmoe`` is a thin ctypes binding with the
same entry-point names.  Importing the package loads nothing; import
``mxfp4_mixture_experts_softmax_gb300.libmoe`` to load the library, which
raises if it is missing (there is no CPU fallback).
"""
