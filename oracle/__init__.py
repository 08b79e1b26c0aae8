"""CPU oracle of the Flint-shaped 4-bit sparse MoE FFN layer.

TEST INFRASTRUCTURE, not product code. Only the test suite, the smoke check
(``__graft_entry__.smoke``) and the CPU-baseline leg of ``bench.py`` may import
it. It is a plain, slow, float64 numpy restatement of what the layer computes,
kept independent of the CUDA path: the two share no code, and neither imports
the other. The seeded input generator
(``bit_quantized_expert_softmax_b300.synth``) is the only thing both consume.
"""
from . import formats, lm_head, moe  # noqa: F401
