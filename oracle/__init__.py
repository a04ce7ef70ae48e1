"""fp64 CPU oracle for the Hogwild! concurrent-attention decode step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or run this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` use it.  It shares no code with the CUDA library (``workload`` only
supplies seeded inputs) and is written from the method's description, not from any kernel:

* ``oracle.rope``      -- rotary position embedding rho(x, p), half-split pairs, fp64.
* ``oracle.cache``     -- the shared cache as a state machine: blocks, paragraph commits, the
                          deterministic page allocator (integers, bit-exact) and the four cache
                          layouts' views (combined, step-wise, contiguous, no-sync).
* ``oracle.attention`` -- the views of each worker and two independent formulations of the
                          concurrent attention: brute force (re-rotate every key at its position
                          in the worker's view) and the method (keys at block-local positions,
                          one query rotation per block, log-sum-exp merge); and the same two
                          for several causal query tokens per worker (``*_mq``).

Source: "Hogwild! Inference: Parallel LLM Generation via Concurrent Attention", summary at
gentlecold.top, sections 4-6 (views, the RoPE identity, the cache layouts), 10 (the no-sync and
step-wise settings of the collaboration scores), 8 (inference flow:
append, attend, commit at step end) and 9 (block-local positions, per-block query rotation,
split work merged by partial-result reduction).
"""
