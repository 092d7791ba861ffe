"""CPU oracle for the exact speculative-decoding verify pass -- TEST INFRASTRUCTURE.

This package is a plain, slow, obviously-correct restatement of what the
verify pass computes, written from the TensorFold pages:

* ``linear``   -- W4 group-quantised linear layer in fp64 (C, ``w4_ref.c``);
* ``affine``   -- MLX-style affine 4-bit linear layer (scale and bias per group);
* ``nvfp4``    -- NVFP4 linear layer (E2M1 codes, E4M3 scale per 16, fp32 global scale);
* ``sampling`` -- keyed Gumbel-max sampling over top-k / top-p candidates;
* ``accept``   -- longest-prefix acceptance of drafts;
* ``moe``      -- top-8 routed W4 SwiGLU experts;
* ``decoder``  -- the attention-free synthetic decoder, serial and drafted;
* ``attention`` -- causal grouped-head attention of verify rows over a KV cache.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import it.  It shares no code with the
CUDA library and never imports the product package; both sides are fed the
same inputs from ``w4_gemm_keyed_gb300.inputs`` by the caller.

Every function with no independent pin says so in its docstring ("parity
unpinned"); the pins live in ``tests/test_oracle_*.py``.
"""

from .linear import w4_linear, half_to_f64, bf16_to_f64, unpack_codes, num_threads  # noqa: F401
from .numerics import bf16_round, bf16_bits_of  # noqa: F401
from . import sampling, accept, moe, decoder, affine, attention, nvfp4  # noqa: F401
