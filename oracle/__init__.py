"""Plain, slow, obviously-correct CPU oracle for the causal video-VAE decoder hot path.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import it: only `tests/`,
`__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py` use it. It shares no code with
the CUDA library (no kernels, headers, helpers or constants) and imports nothing from it.

Everything here is numpy in fp64 (the pages fix fp32 only for the phase-weight sums, which the
oracle then does in fp32), following the statements of the method on the pages:
  * WanGP `shared/kernels/group_norm_silu.py` (module docstring and `_apply_kernel`):
    silu(group_norm(x)) with population variance, eps inside the square root, one rounding.
  * FastVideo `wan22_vae_decode/solution/binding.cpp`:
    - `Decoder::conv` and `Decoder::resnet`: the causal 3x3x3 convolution whose padded input is
      the carried cache frames followed by the chunk, the cache update to the last two padded
      input frames, bias and residual added before the output rounding;
    - `prepare()`: the nearest-x2 + 3x3 = four 2x2 phase-convolution weight transform, summed in
      fp32 and stored in bf16;
    - `decode_video`: the history crosses chunks in the cache, so the result does not depend on
      the chunk size.

Every function is pinned by a `-m "not gpu"` test against something other than itself (brute
force, a library routine, a closed form or an invariant); see `tests/test_oracle_*.py`.
"""
from .reference import *  # noqa: F401,F403
