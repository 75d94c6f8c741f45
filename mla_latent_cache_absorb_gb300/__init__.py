"""GB300-native MLA absorbed decode over a compressed latent KV cache.

The compute lives in the C-ABI library `libmla.so` (hand-written CUDA for sm_103a);
`binding` marshals arguments to it through ctypes. `synth` draws seeded inputs.
"""
