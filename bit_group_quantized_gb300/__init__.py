"""GB300-native 4-bit / 2-bit group-quantized MoE decode path.

The compute lives in ``libbgq.so`` (CUDA kernels for sm_103a behind a C ABI,
declared in ``include/bgq.h``); :mod:`.lib` is its thin ctypes binding and
:mod:`.synth` the seeded input generator. Importing the package loads
neither, so the generator can be used on machines without the library.
"""
