"""Plain, slow CPU oracle of the tiered (BF16 / INT2 / evicted) KV-cache decode path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.
It shares no code with the CUDA path; its only input dependency is the
seeded generator module ``qe_inputs`` (which holds none of the method's
arithmetic).

Floating point is float64 except where the pages fix another precision:

* the quantizer (HqeKV reading notes, §2.3 eq. (2)) runs in float32, the
  precision the CUDA packer decides codes in, so codes and min/scale
  parameters can be compared bit for bit;
* accumulated window scores are stored in float32, as the H2O page
  (§3.1 and §5.1) asks of score storage; each step's increment is
  computed in float64 and rounded once before the float32 add;
* routing decisions compare those float32 scores.

Modules
-------
quant      eq. (2) uniform min/scale quantizer and KIVI's asymmetric axes
budget     byte accounting, eq. (3) tier capacities, per-workload capacity rules
router     candidate pool eq. (4), greedy TopK assignment eq. (5)
attention  decode attention over the accessible mixed set, per-window mass
qevict     per-(batch, layer, KV head) state machine: append, decode step, route
h2o        token-level H2O step (the heavy-hitter special case of the router)

Parity status: every function is pinned by a ``-m "not gpu"`` test
(``tests/test_oracle_*.py``) except the long-run trajectories of the
32-layer workloads, whose tier sequences beyond the invariants are
"parity unpinned" (checked only against the CUDA path).
"""
