"""CPU oracle for the Muon optimizer step -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously correct NumPy restatement of the Muon
step (Nesterov momentum, quintic Newton-Schulz orthogonalisation, parameter
update).  It exists to check the CUDA path and to serve as the timed CPU
baseline.  Only the test-suite, the smoke check and the benchmark's CPU-baseline
and reference legs may import it; the product path never does, and it shares no
code with the CUDA kernels.

Source of the method:
  page "深入解析KellerJordan/modded-nanogpt中的训练架构与优化技术"
  (reposource.net, an annotated walk-through of modded-nanogpt's train_gpt.py),
  sections "Muon优化器：动量正交化技术" (the Muon class and its defaults) and
  "Newton-Schulz正交化" (the function zeropower_via_newtonschulz5 and its
  coefficients).

Three steps are not printed on that page; the readings taken here are stated in
``oracle.muon`` next to the code that takes them.

``oracle.fp8`` restates the FP8 scaled matrix multiplication (E4M3 forward,
E5M2 gradients, BF16 results) that the same walk-through page describes in
section "自定义FP8矩阵乘法实现"; its readings are stated there.

``oracle.adam`` restates the Adam step with cautious weight decay that the page
on the modded-nanogpt record "2026-06-11_RecursiveFromBest" (lqnn.cn,
news/184262, section "3.3 bigram 与 value-embedding 银行上的 C-Optim / 谨慎
Adam") describes for the embedding-type banks; its readings are stated there.

Pin status: every public function is pinned by the CPU tests
(closed form via SVD, invariants, brute force in exact rational arithmetic,
bit-exact bf16 rounding against an independent routine; for Adam: closed
forms, torch.optim.Adam / AdamW special cases, hand-worked mask values; for
FP8: bit-exact casts against torch's float8 conversions and a bit-field
decoding of all 256 codes, exact products of representable operands, power-of-
two scale invariance, brute force in rational arithmetic).
"""

from .adam import ADAM_DEFAULTS, adam_constants, adam_step, cautious_mask
from .fp8 import FP8_FORMATS, fp8_mm, fp8_mm_backward, quantize, round_to_fp8
from .bf16 import round_to_bf16, BF16_MAX
from .muon import (
    NS_COEFFS,
    NORM_EPS,
    MUON_DEFAULTS,
    momentum_update,
    orient,
    normalise,
    ns_gram,
    ns_poly,
    ns_update,
    ns_iteration,
    ns_iteration_parts,
    newton_schulz5,
    muon_step,
)

__all__ = [
    "FP8_FORMATS",
    "fp8_mm",
    "fp8_mm_backward",
    "quantize",
    "round_to_fp8",
    "ADAM_DEFAULTS",
    "adam_constants",
    "adam_step",
    "cautious_mask",
    "round_to_bf16",
    "BF16_MAX",
    "NS_COEFFS",
    "NORM_EPS",
    "MUON_DEFAULTS",
    "momentum_update",
    "orient",
    "normalise",
    "ns_gram",
    "ns_poly",
    "ns_update",
    "ns_iteration",
    "ns_iteration_parts",
    "newton_schulz5",
    "muon_step",
]
