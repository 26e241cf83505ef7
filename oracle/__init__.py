"""CPU float64 oracle for the owner-local Muon optimizer step (test infrastructure only).

This package is the reference the CUDA path is checked against.  It is plain, slow and
written for a reader to check by eye against the method's description: numpy float64, one
library matmul per product, no blocking, fusion or reordering.  It shares no code with the
CUDA path, the C-ABI library or its Python binding, and imports none of them.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  The product path never calls it and never falls back to it.

Source: "MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding"
(academ.us/article/2607.05895).
  * ``plan``   — owner-shaped placement and the greedy owner planner (§3, §4.1, §4.2).
  * ``muon``   — owner gradient deposit, Nesterov momentum, Newton–Schulz, scaled update
                 with decoupled weight decay (§2, §3, §4.4, §5.1, §5.3).
  * ``adamw``  — the coordinate-wise AdamW step of the packed non-2D tail (§3, §5.1).
  * ``step``   — several optimizer steps of a whole owned set, as lists of matrices.
  * ``repack`` — canonical parameter axis <-> owner shards (§4.2, §4.4).
  * ``shampoo`` — owner Shampoo: statistics, inverse fourth roots, update (§5.7).
  * ``soap``   — owner SOAP: Adam in the eigenbasis of the Shampoo statistics (§5.7).

Pins (checked by ``tests/test_oracle_pins.py`` against things other than this code):
  plan   — invariants, the list-scheduling bound, hand-worked assignments, brute force;
  reduce — exact sums of integer-valued contributions;
  momentum — the constant-gradient closed form;
  Newton–Schulz — the singular-value identity against ``numpy.linalg.svd`` and the scalar
           quintic, 1x1 / row / diagonal special cases;
  update — closed forms with O = 0 and with a known O;
  AdamW  — a hand-worked single-element run and the first-step identity.
  repack — round trips, hand-worked layouts, reshard = direct pack;
  Shampoo — closed-form roots (diagonal, Q diag Q^T), the scalar and rank-one steps,
           orthogonal invariance;
  SOAP   — the 1x1 case against the hand-worked AdamW run, diagonal gradients against the
           coordinate-wise AdamW, the rank-one closed form, orthogonal equivariance,
           transpose symmetry and eigenvector-sign invariance.
No function here is "parity unpinned".
"""
