"""Python binding of libsoup: the streamed NF4 LoRA step on sm_103a.

Argument marshalling only — every step of the path runs in the CUDA library, loaded from
``libsoup.so`` next to this file.  There is no CPU fallback: if the library is missing,
importing :mod:`nf4_dequant_gemm_blockwise_b300.api` raises.  Build it with
``python -m nf4_dequant_gemm_blockwise_b300.build``.
"""
