"""FP8 weight-only (w8a16) decode GEMV for GB300 (sm_103a).

y[m,n] = bf16(scale[n] * sum_k bf16(W[n,k]) * x[m,k]) with W an E4M3fn plane
and one fp32 scale per row (ATOM pull request #2980,
Summary and Changes); bf16 planes run through the same entry point.

The compute path is the C-ABI library ``libw8.so`` (include/w8.h) built from
``csrc/``; ``fp8_weight_only_w8a16_gb300.w8`` is its thin ctypes binding.
Importing the package does not load the library; importing ``.w8`` does, and
raises if the library is missing.
"""
