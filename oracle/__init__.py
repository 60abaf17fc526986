"""CPU oracle for the drafter-sampling hot path (TEST INFRASTRUCTURE ONLY).

A plain, slow, fp64 restatement of what the hot path computes, written from
the pages that define the method:

* "VocabTrim: Vocabulary Pruning for Efficient Speculative Decoding in LLMs"
  (arXiv 2506.22694): Algorithm 1 (token-frequency counter), eq. (1)
  (Top-K vocabulary and the trimmed LM head W[Top-K(c,k),:]), Algorithm 2
  (drafting through the trimmed head and the index mapper T_{d->t}).
* "Speculative decoding" (SelfMadeQuant glossary), section "Why a rejection
  needs a special draw": acceptance min(1, p/q) and the residual
  norm(max(p-q, 0)), plus the two-token worked example.
* "A rejection rule keeps speculative decoding's output exact" (the nightly
  build), sections "Extending the rule from one token to a drafted run" and
  "What draft accuracy buys": left-to-right block verification, the bonus
  draw, beta = sum min(p, q), and E[#tokens] = (1-alpha^(gamma+1))/(1-alpha).

Only the test suite, ``__graft_entry__.smoke()`` and the bench's CPU-baseline
leg may import this package.  It shares no code with the CUDA library and the
library never calls it.

Every public function is pinned by ``-m "not gpu"`` tests against facts the
pages or the mathematics fix (none is "parity unpinned"):

* inverse_cdf            strict edges on hand-worked weights, zero-weight bins
                         never drawn, last-positive fallback, chi-square of
                         200k Philox draws (tests/test_oracle_sampling.py)
* softmax                closed forms (0, ln 3) -> (1/4, 3/4), at T=1/2 ->
                         (1/10, 9/10); shift invariance
* acceptance_probability the glossary's two-token table (0.75, 1)
* residual_weights       the glossary's residual (0, 1)
* verify                 exact integration over its uniforms: two-token final
                         mass (0.6, 0.4) and the naive-redraw control
                         (0.72, 0.28); emitted tokens and pairs follow p on
                         V=3 (gamma=2), V=18 (gamma=1) and with temperature;
                         survival probability = sum min(p, q); mean block
                         length = (1-beta^(gamma+1))/(1-beta) at constant beta;
                         chi-square of a 20k-block toy chain, and rejection of
                         the planted naive redraw (tests/test_oracle_verify.py)
* token_histogram        hand-worked fixtures, collections.Counter, sum = N
* top_k                  hand-worked ties, Python sorted() on (-count, id)
* ranking / top_p /      hand-worked counts; brute force over every prefix
  min_count              length; Top-P at P = 1 keeps every counted id; the
                         selections agree with top_k at their own K
                         (tests/test_oracle_select.py)
* trim_head              bit-for-bit rows, inverse map, head sizes of
                         VocabTrim's Tables 1-3
* draft_logits           exact rational dot products; one-hot hidden
* draft_step             two-token softmax and sampling edges; equality with
                         the masked full-vocabulary head; chi-square of draws
                         (tests/test_oracle_vocabtrim.py)
* argmax_lowest          hand-worked ties; numpy argmax on distinct values
* draft_step_greedy      exact rational dot products; the sampling draft at a
                         vanishing temperature
* verify_greedy          lossless: chained greedy speculative decoding emits
                         exactly the target's own greedy stream on the toy
                         tables; equals the stochastic verify at a vanishing
                         temperature for any uniforms; hand-worked blocks
                         (tests/test_oracle_greedy.py)
* verify_tree_greedy     a chain equals verify_greedy; the deepest accepted
                         path equals the best root-to-leaf chain (brute
                         force); lossless tree decoding on the toy tables;
                         hand-worked trees and depth ties
* draft_topk             exact integer logits and ties; exp(log q) equals
                         the pinned draft_step's q; k = 1 is the greedy draft
                         (tests/test_oracle_tree.py)
"""
from .sampling import inverse_cdf, InverseCdfResult  # noqa: F401
from .vocabtrim import (token_histogram, top_k, trim_head, bf16_to_f64,  # noqa: F401
                        draft_logits, draft_step, BadInput, ranking, top_p, min_count)
from .speculative import (softmax, acceptance_probability, residual_weights,  # noqa: F401
                          verify, VerifyResult)
from .greedy import (argmax_lowest, top2_gap, draft_step_greedy, verify_greedy,  # noqa: F401
                     GreedyResult)
from .tree import verify_tree_greedy, draft_topk, TreeResult  # noqa: F401
