"""CPU oracle for the ragged_dot (MoE grouped GEMM) hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (no kernels, headers, helpers or tables).

Every function is a plain, slow restatement of what the pages define, in
float64 unless the pages fix another precision:

* ``ragged.ragged_dot``            -- grouped forward with group_offset and limit
* ``ragged.ragged_dot_trans_rhs``  -- the trans_rhs form used for dx
* ``ragged.ragged_dot_trans_rhs_glu_bwd`` -- dx of the down projection followed
                                      by the SiLU-GLU backward
* ``ragged.trans_ragged_dot``      -- per-group weight gradient x^T y
* ``ragged.trans_ragged_dot_f32``  -- the same in f32, optionally accumulated
* ``ragged.ragged_dot_adjusted``   -- the boundary-absorbing formulation of
                                      fast_ragged_dot (second formulation)
* ``glu.*``                        -- SiLU-GLU forward/backward in float64 and
                                      as the float32 op sequence
* ``unsort.unsort_bwd_rows``        -- weighted gradient and routing-weight row dot
* ``bf16.*``                       -- bf16 rounding and ulp helpers

Parity status: every function here is pinned by tests under ``tests/``
(brute force on tiny inputs, closed forms, invariants, finite differences);
none is "parity unpinned".  The pages print no numeric input/output example,
so no pin comes from printed values.
"""
from . import bf16, glu, ragged, unsort  # noqa: F401
from .ragged import (  # noqa: F401
    group_bounds,
    ragged_dot,
    ragged_dot_adjusted,
    ragged_dot_trans_rhs,
    ragged_dot_trans_rhs_glu_bwd,
    trans_ragged_dot,
    trans_ragged_dot_f32,
)
from .glu import (  # noqa: F401
    glu_bwd_f32,
    glu_bwd_f64,
    glu_fwd_f32,
    glu_fwd_f64,
)
