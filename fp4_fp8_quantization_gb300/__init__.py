"""GB300-native grouped mixture-of-experts low-precision kernels.

``moeq``  - Python binding of the C ABI (libmoeq.so, include/moeq.h).
``synth`` - seeded synthetic MoE-shaped inputs.
``build`` - nvcc build of libmoeq.so for sm_103a.
"""
