"""GB300 speculative-decoding verify round.

- `spec`   : ctypes binding of the C ABI in include/spec_verify.h (loads
             libspecverify.so; raises if it has not been built).
- `synth`  : seeded synthetic inputs (weights, prompts, uniforms, Dirichlet draws).
- `build`  : compiles the CUDA library for sm_103a in place.

Importing the package does not load the CUDA library; `spec` does.
"""
