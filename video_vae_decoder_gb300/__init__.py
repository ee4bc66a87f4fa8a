"""GB300-native (sm_103a) hot path of a causal 3D video-VAE decoder: GroupNorm+SiLU, the causal
3x3x3 convolution with its carried temporal cache, the causal ResBlock, and the nearest-x2
upsample executed as four 2x2 phase convolutions, behind the C ABI declared in include/wan.h.

`binding` loads the in-tree shared library (built by `build.build()`) and marshals arguments;
every step of the computation runs in the library's CUDA kernels.
"""
