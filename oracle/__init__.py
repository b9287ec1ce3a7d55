"""CPU oracle (test infrastructure only): see ``oracle.tq_oracle``.

Parity status per function (what pins it, from tests/test_oracle.py):
  hadamard / rotate / unrotate    pinned: scipy's Sylvester Hadamard, orthonormality, inverse
  lloyd_max_gaussian / codebook   pinned: closed form at 1 bit, Max (1960) table, optimality
                                  conditions by numerical quadrature, Monte-Carlo MSE
  quantize                        pinned: brute-force nearest centroid
  turbo_encode / turbo_dequant    pinned: hand-derived d=2 case, QJL sign rule with S = I,
                                  distortion vs Lloyd MSE, compressed-domain score identity
  qjl_stage                       pinned: through turbo_encode; hand-derived d=2 case with another
                                  index and a non-symmetric S; linearity in the index
  qjl_inner_product_estimate      pinned: Monte-Carlo unbiasedness and variance bound
  q8_0_encode / q8_0_dequant      pinned: exact integer blocks, half-away ties, error <= delta/2
  minmax_encode / minmax_dequant  pinned: the pages' worked examples (codes 0/8/15, 6/6)
  decode_attention                pinned: single token, identical keys, tau = 0, GQA mapping,
                                  scipy softmax
  compressed_scores               pinned: equals scale <q, k~> of the dequantised cache
  prefill_attention               pinned: a one-token chunk equals decode_attention, brute-force
                                  scalar loops on a tiny input, causality
"""
