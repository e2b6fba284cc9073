"""CPU oracle for the persistent decode megakernel -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import, call, link or execute anything in this package.
The product path (the ``persistent_megakernel_decode_gb300`` package and its
CUDA library) never imports it and shares no code with it.

Parts:

* ``rules``   -- the planner rules written out plainly: MPK's gcd event
  partition with the fork/join lcm normalisation, MegaRTP's four pairing
  strategies, task linearisation with contiguous successors, static queue
  assignment with NoOp padding, expected final counter values.
* ``sim``     -- a queue simulator: deadlock check over in-order per-worker
  queues and a random-interleaving executor that runs real tile math.
* ``tail``    -- the wave-quantisation (tail) arithmetic of a kernel-per-op run.
* ``forward`` -- ctypes front end of ``forward.c``: a plain per-op decoder
  forward (fp64 accumulation, or fp32 for timing) and the GLM-style
  pre-attention block.

Parity status of each function is stated in its docstring ("pinned by ..." or
"parity unpinned").
"""
