"""CPU oracle for the DSpark draft/verify hot path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import
anything here.  The product (the CUDA library and its Python binding) never
imports, links or runs this package, and shares no code with it.

Everything is plain numpy in float64 (integers exact), written step by step
from the pages that define the method, each function citing its passage:

  * "DSpark implementation and evaluation" (ggaaooppeenngg.github.io):
    §2.2 Sequential Markov Sampling, §3 Markov Head structure, §4 draft step,
    §5 reduced draft vocabulary and verification with the draft's Gumbel noise.
  * "Speculative decoding: from zero to DSpark" (bittide.aicompass.dev):
    §2 the loop and its lossless property, §6 scheduling by expected
    throughput and the calibrated confidence head, §7 running in a real engine.
  * "xserv/docs/25-speculative-methods-comparison.md": §2 greedy verification,
    §3.2 the draft-to-target id table.

Where the pages are silent (the random-number counter layout, the uniform
mapping, the fixed-point resample, the objective's exact form) the oracle
takes one plain reading; the same readings are implemented independently by
the CUDA path.

Pins: every function here is checked by ``tests/test_oracle_*.py`` against
closed forms, library routines (cuRAND's host Philox generator, numpy/scipy),
brute force on tiny inputs and statistical laws -- never against the CUDA path.
"""
from .philox import philox4x32_10, philox_words, uniform_from_word, gumbel_from_word
from .draft import draft_logits, markov_sample, markov_bias
from .verify import verify, acceptance_probability_exact
from .schedule import schedule, survival_chain
from .greedy import verify_greedy, row_argmax
from .confidence import confidence
from .reduced_vocab import map_to_target, markov_sample_reduced
from .verify_logits import verify_from_logits, draft_distributions, draft_lse, residual_gumbel
from .verify_gumbel import verify_gumbel, target_gumbel_tokens

__all__ = [
    "philox4x32_10", "philox_words", "uniform_from_word", "gumbel_from_word",
    "draft_logits", "markov_sample", "markov_bias",
    "verify", "acceptance_probability_exact",
    "schedule", "survival_chain",
    "verify_greedy", "row_argmax", "confidence", "map_to_target", "markov_sample_reduced",
    "verify_from_logits", "draft_distributions", "draft_lse", "residual_gumbel",
    "verify_gumbel", "target_gumbel_tokens",
]
