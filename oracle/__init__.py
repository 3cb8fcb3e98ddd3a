"""CPU oracle for the blockwise attention + FFN layer.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's ``smoke()`` check and
the CPU-baseline leg of ``bench.py`` may import anything from here; the
product path (the CUDA library and its Python binding) never does.

* :mod:`oracle.ref` -- plain, materialised fp64 NumPy definition of the layer,
  forward and analytic backward, plus a blockwise (online-softmax) fp64
  variant used only to pin the definition against the method's own claim of
  exactness.
* :mod:`oracle.tiny` -- scalar-loop forward for tiny shapes (cross-check).
* :mod:`oracle.accounting` -- the pages' parameter / activation / FLOP
  accounting formulas.
* :mod:`oracle.sampled` -- row-sampled forward and sparse-upstream-gradient
  backward for sequence lengths where the dense oracle is too slow.
* :mod:`oracle.lm_loss` -- the language-model loss after the last layer
  (mean token cross-entropy through the vocabulary projection) and its
  position- and vocabulary-blocked forms, for the blockwise-loss row that
  comes next.
* :mod:`oracle.stack` -- a stack of layers trained with a checkpoint every k
  layers (the multi-layer row that comes next).
* :mod:`oracle.sharded` -- one layer sharded by sequence position over P
  ranks (zigzag rows, K/V all-gather, dK/dV reduce-scatter, weight-gradient
  all-reduce), with the collectives passed in; the tests run it on gloo
  ranks on CPU.
"""
