"""Oracle: a plain, slow CPU restatement of one DFlash + DDTree speculative step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it.  The CUDA library never calls it and it
never calls the CUDA library; the two share no code.  Inputs come from ``synth``.

Arithmetic is float64 with numpy (a matrix product, a sort and ``exp``/``log`` are
the only library steps), except where the method itself fixes float32: the
log-probabilities handed to the tree builder and the tree's prefix scores, which are
float32 sums exactly as the CUDA path forms them, so tree topology can be compared
bit for bit.

Sources, cited by page and section throughout:
  [DFlash]  "DFlash: Block Diffusion for Flash Speculative Decoding 논문 정리"
            (honbul.tistory.com/178), a summary of Chen, Liang, Liu, arXiv 2602.06036.
  [DFlash-news]  darkpulse.kr/?p=2484, a news summary of the same method.
  [DDTree]  bluediary8.tistory.com/1288, a summary of Ringel & Romano,
            "Accelerating Speculative Decoding with Block Diffusion Draft Trees".

Parity pins (see tests/test_oracle_*.py):
  ddtree.build_tree       brute-force top-B enumeration, prefix-closed optimality,
                          Monte-Carlo acceptance identity.      PINNED
  ddtree.build_chain      exhaustive search over all token sequences (the chain is
                          the best sequence, ties to the lowest ids); equals build_tree
                          with B = D when each position has a dominant token.  PINNED
  ddtree.log_softmax      normalisation, shift invariance, scipy.     PINNED
  ddtree.topk_sorted      heapq.nlargest on the same key.            PINNED
  model.rms_norm / rope   closed forms (unit RMS, rotation, relative position). PINNED
  model.attend            hand-worked 3x5 case (tests/golden).        PINNED
  verify.tree_attention   equals causal attention over each root path. PINNED
  verify.greedy_walk/compact  hand-built trees.                        PINNED
  step.spec_generate      token-identical to step.greedy_generate (losslessness). PINNED
  model.moe_route / moe_block  (mixture-of-experts target) reduction to the dense layer
                          with one expert, brute force over expert subsets, relabelling
                          invariance, a torch-library formulation, tree rows = sequential
                          decode.                                      PINNED
  sample.draw / sampler   (temperature verification, a reading: the pages state no rule)
                          fmix32 bijection, uniform and Gumbel laws of the noise, draw
                          frequencies = softmax(logits / T), small-T limit = argmax;
                          step.spec_generate with drawn choices token-identical to plain
                          sampling (losslessness at temperature 1).    PINNED
  model.layer_forward     pinned only through the invariants above: the pages
                          print no layer equations or values (a Qwen3-style
                          pre-norm layer is the stated reading).
"""
