"""CPU oracle for one frame of the codec-TTS depth decoder.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import, call
or run anything in this package. The product path (the C-ABI library and its
Python binding) never does, and shares no code with it: the only module both
sides use is ``synth`` (seeded input generators, no arithmetic of the method).

Plain numpy, float64 unless a step decides an integer from floating point (the
draw, float32 like the kernel). Every function cites the passage it follows.

Modules:
* ``philox``  -- Philox4x32-10 and the per-vocabulary uniforms of a draw.
* ``draw``    -- temperature / top-k / top-p / Gumbel-max draw of one row.
* ``frame``   -- the whole frame (input projection, 5-layer GQA transformer
  over 16 depth positions, 15 heads and draws, 16 embedding steps), with a
  float64 mode, a bf16-operand mode and teacher forcing.
* ``plan``    -- the frame's phase sequence and its weight bytes in closed form.

Pins (tests/test_oracle_*.py, run with ``-m "not gpu"``): every function here
is checked against something other than itself -- hand-computed values,
closed forms, invariants, library routines (torch functional ops, triton's
Philox under its CPU interpreter) and brute force on tiny inputs. No function
is left unpinned.
"""
from . import philox, draw, frame, plan  # noqa: F401
from .frame import run_frame, bf16_round, rms_norm, rope, silu, attention  # noqa: F401
from .draw import draw_detail  # noqa: F401
