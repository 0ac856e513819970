"""CPU oracle for the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, deliberately
unoptimised restatement of what the verify step computes.  It exists so that
the CUDA library can be checked against something that a reader can compare
with the source pages by eye.  Only the test-suite, the smoke check and the
CPU-baseline leg of the benchmark may import it; the library never does, and
this package imports nothing from the library.

Sources (cited by page title and section throughout):

* "Speculative decoding on RDNA" (hipfire learn page): §01 the speculative
  window and the at-least-one-token rule, §02 greedy acceptance and the
  row-count-invariant projection, §03 rejection sampling and the sampler
  policy, §04 per-row penalty histories.
* "One RDNA4 verify pass has slack for about two dozen speculative tokens"
  (zolotukhin.ai blog): token-tree verify, "Spend the budget on a tree".
* "feat(dflash): developer-only online draft tuning" (hipfire PR #820):
  naive sampling verify for deterministic drafts ("spec step" listing notes),
  top-K tie/NaN/-inf byte identity.

Modules:
  philox  -- Philox4x64-10 counter-based generator (Salmon et al., SC'11).
  vexp    -- the deterministic exponential used by the policy (Cody-Waite
             reduction plus a Taylor polynomial), IEEE +,-,x only.
  verify  -- projection, histories, penalties, pool, policy, draws and
             acceptance (chain greedy, chain rejection sampling, token tree
             greedy, naive sampling descent), the window and the batched form.

Parity status: every function here is pinned by a CPU test against something
other than itself (numpy's Philox, libm, exact rationals, brute force,
scipy's softmax, exact enumeration, a chi-square with a failing control).
The one thing that is not pinned is the summation order inside the GPU
projection, which only has to agree with itself across row counts.
"""
