"""CPU oracle for the split-backward MLP stage and its pipeline orderings.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code with the CUDA library
(``split_backward_gemms_gb300``); the two meet only through the seeded input
generators in ``split_backward_gemms_gb300/inputs.py``, which hold none of the
method's arithmetic.

Modules
-------
``block``      fp64 numerics of one stage's MLP block: the forward F, the
               input-gradient B and the weight-gradient W, plus the
               single-linear special case and an fp64 pipeline chain.
``schedules``  1F1B / ZB-H1 / ZB-H2 event-graph generators (a list-scheduling
               simulator), the heuristic ZB-1p / ZB-2p scheduler, an op-list
               validator and a timed-trace checker built from the event
               graph's dependency rules, bubble metrics, the closed forms and
               the activation-memory ledger.
``interleaved`` two-chunk orderings: interleaved 1F1B (cyclic assignment)
               and ZB-V (V-shaped), their simulator, the gap-free search and
               integer program, and the mapping onto the chain of virtual
               stages.
``optimizer``  AdamW, its algebraic inverse and the staged-reduce
               post-update validation of the stages' optimizer steps.

Sources are the three web pages on zero bubble pipeline parallelism:
  * "Zero Bubble Pipeline Parallelism" (paper-graph-ui summary of arXiv
    2401.10241), cited as [ZB-PP summary] with its section / table / equation;
  * "Zero-Bubble Pipeline Parallelism, Proven" (jpcasabianca.com journal),
    cited as [ZB proven];
  * "Pipeline Schedules: GPipe, 1F1B and Zero Bubble" (neelmishra.github.io),
    cited as [Pipeline schedules].

Every function is pinned by a ``-m "not gpu"`` test against something other
than itself (closed forms, finite differences, textbook special cases, the
worked example on [ZB proven], brute force on tiny inputs).  No function here
is "parity unpinned".
"""
