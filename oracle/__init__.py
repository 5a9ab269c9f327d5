"""CPU oracle for the rank-local ZeRO optimizer step — TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct numpy implementations of what the GPU path computes, each
written from the source pages' own statement of the method:

* ``oracle.layout``  — the flat bucketed shard layout (deg/zero.py, ZeroMaster: class
  docstring, ``__init__`` bucket construction, ``_segments``/``_pieces``).
* ``oracle.bf16``    — round-to-nearest-even fp32 -> bf16 (deg/zero.py, ``gather_params``:
  the shard rounded to the compute dtype).
* ``oracle.adamw``   — per-tensor AdamW with decoupled weight decay and per-step bias
  correction, in an exact-op-order fp32 mode and an fp64 mode (dmuon PR #16, "foreach
  AdamW" commit: op order; DeepSpeed PR #9021, grad_scale-on-load commit; bluscript_zero_ckpt.cpp,
  ZeroConfig hyper-parameters and the fp32-master note).
* ``oracle.clip``    — Σg², global norm, clip coefficient, clipped / found_inf
  (deg/zero.py ``grad_sq_norm``; bluscript_zero_ckpt.cpp, global clip block; dmuon PR #16,
  sync-free clip stats commit).
* ``oracle.ns``      — Muon's quintic Newton-Schulz in fp64 (bluscript_zero_ckpt.cpp, the
  ShardedMuon design note: ``X <- aX + (bXX' + c(XX')^2)X``).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm
may import this package. The product path (the ``zero_sharded_optimizer_flat_gb300``
package and its CUDA library) never imports, links or runs anything here, and this package
never imports the product. The two share no code; inputs come from ``workloads``.

Every function is pinned by ``-m "not gpu"`` tests against something other than itself
(closed forms, brute force, library routines, invariants). Nothing here is "parity unpinned".
"""
