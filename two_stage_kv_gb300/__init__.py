"""GB300 (sm_103a) two-stage compressed decode attention (RocketKV hot path).

Submodules: `rkv` (ctypes binding of include/rkv.h), `pipeline` (device
buffers and call sequences built on the binding), `synth` (seeded synthetic
inputs), `build` (nvcc build of the in-tree library).  Importing the package
does not load the CUDA library; the first binding call does, and raises if it
is missing.
"""
