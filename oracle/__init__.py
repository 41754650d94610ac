"""CPU oracle for draft branch attention — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct numpy (fp64) statement of what the branch
attention path computes, written from the pages about "Online Draft
Co-Training for Speculative Decoding in Large-Scale, Long-Context RL
Post-Training" (arXiv 2609.07108).  It shares no code with the CUDA path and
never imports it.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it; the product path never calls
it and has no CPU fallback.

Modules
-------
keysets     which keys each branch query attends (the branch mask)
attention   dense masked softmax attention and its gradients, full and sampled
merge       the online-softmax log-sum-exp merge (Eq. 2)
zigzag      packed zigzag chunking, virtual-rank ownership, ring schedule, Eq. 3
decomposed  main-ring partials + rank-local branch part + Eq. 2 (self-check path)

Pins (see ``tests/test_oracle_*.py``): uniform-attention key-set counting
against closed forms, a torch fp64 SDPA cross-check with an independently
built mask, finite differences, exact gradient invariants, the decomposition
identity to 1e-10, and the hand-worked fixtures under ``tests/golden/``.
No function here is parity-unpinned.
"""

from . import keysets, attention, merge, zigzag, decomposed  # noqa: F401
