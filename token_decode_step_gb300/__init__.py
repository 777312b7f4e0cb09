"""GB300 (sm_103a) one-token decode step of a Qwen3-style dense decoder.

The product is the C-ABI library ``libdec.so`` (include/dec.h) built from
``csrc/``; ``dec`` is its ctypes binding and ``torch_glue`` marshals PyTorch
tensors into it.  Build with ``token_decode_step_gb300.build.build()``.
"""
