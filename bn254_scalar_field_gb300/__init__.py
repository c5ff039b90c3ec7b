"""GB300 (sm_103a) library for the Groth16 quotient-evaluation (H) path over BN254 Fr.

The compute path is the CUDA library libg3h.so behind the C ABI in include/g3h.h;
``g3h`` is its ctypes binding and ``build`` compiles it in-tree. ``synth`` draws the
seeded synthetic inputs.
"""
