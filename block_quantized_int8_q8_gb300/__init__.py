"""Block-quantized int8 MMQ for GB300 (sm_103a).

`api` binds the CUDA library (libmmq_gb300.so, C ABI in include/mmq.h); `synth` draws seeded synthetic
inputs in the library's byte layouts.  Importing the package does not load CUDA; the first call into
`api` loads the library and raises if it is missing.
"""
