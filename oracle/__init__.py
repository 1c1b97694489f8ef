"""Plain fp64 CPU oracle for the sequence-parallel DiT attention hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or runs
this package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may use it.  It shares no code with the CUDA library under
``sequence_attention_gb300/`` and imports nothing from it.

The oracle writes each operation out as its plain definition, in float64 for
all floating-point arithmetic, with numpy as the only numerical library:

* ``attention``   -- softmax(Q K^T * scale) V with the row log-sum-exp,
                     the partial over one key chunk, and the log-sum-exp merge
                     of several partials (SGLang Diffusion "Parallelism
                     Overview", sections "What happens to the shapes" and
                     "Constraints"; edge-dit.cpp "Parallel execution",
                     Ulysses sequence parallelism).
* ``layout``      -- the balanced uneven sequence split, head padding and
                     the all-to-all counts/displacements (edge-dit.cpp,
                     SPSequenceSplit and SPAllToAll4DLayout; cache-dit
                     "Context Parallelism", UAA and "Any Head Num").
* ``ulysses``     -- the sequence<->head all-to-all as an explicit index
                     permutation (edge-dit.cpp packed QKV and head-to-sequence
                     paths; SGLang Diffusion "The Ulysses transport").
* ``cfg``         -- p_uncond + g * (p_cond - p_uncond) (edge-dit.cpp,
                     classifier-free guidance).
* ``usp``         -- Ulysses inside, ring outside, composed end to end
                     (cache-dit "USP: Unified Sequence Parallelism").
* ``numeric``     -- round-to-nearest-even conversions to bfloat16/float16.
* ``fp8``         -- the e4m3 wire of Q, V and O with one scale per
                     (token, head) (cache-dit "Context Parallelism", Async
                     FP8 Ulysses Attention).
* ``rope``        -- rotary embedding of the receive preparation and the
                     joint text+image sequence (edge-dit.cpp, receive
                     preparation and paired text/image streams).

Every function is pinned in ``tests/test_oracle_*.py`` to closed forms,
invariants, library routines or brute force; none is "parity unpinned".
"""

from . import attention, cfg, fp8, layout, numeric, rope, ulysses, usp  # noqa: F401
