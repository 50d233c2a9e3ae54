"""GB300 (sm_103a) causal grouped-query attention step: qkv split, Q/K
RMSNorm, RoPE, KV append and causal GQA, for ragged prefill and split-KV
decode, behind the C ABI in include/attn.h (and token sampling, in
include/sample.h).

Modules: ``attn`` (ctypes binding of libattn.so), ``step`` (device upload
and the packed prefill + decode call sequence), ``inputs`` (seeded synthetic
inputs), ``build`` (nvcc build of libattn.so).  Nothing is imported here, so
that ``inputs`` can be used without loading the CUDA library.
"""
