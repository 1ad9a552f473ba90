"""CPU oracle for the TurboQuant hot path: plain, slow, fp64, obviously correct.

This package is TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
it.  The product path (``compressed_kv_cache_02_b300``) never imports, links or
executes anything here, and this package imports nothing from the product: the
two share no code.  The only module both sides use is the seeded input generator
``compressed_kv_cache_02_b300.inputs``, which draws synthetic data and holds
none of the method's arithmetic.

Everything is numpy in float64.  Library primitives (matmul, QR, searchsorted,
lexsort, the regularised incomplete beta function) serve as single steps; there
is no blocking, fusion or reordering beyond what each docstring states.

Citation legend (the source pages, by title and section):

* [juejin §2]  juejin.cn post 7621817220135075850 (a reading of the Google
  Research blog and arXiv:2504.19874), section 二 "TurboQuant 的两段式：先
  PolarQuant「塑形」，再 QJL「收口误差」": random rotation, scalar quantization
  with most of the bit budget, ~1 bit of QJL on the residual, asymmetric
  estimator with a high-precision query.
* [juejin §3]  same post, section 三 "材料勘读": attention logits over the KV
  cache (4-bit vs 32-bit keys on H100), GloVe d=200 Recall@1@k search.
* [juejin §4]  same post, section 四 "研究论文里多出来的「硬句子」":
  data-oblivious, online, near-optimal MSE and inner-product distortion.
* [freelamp PQ]   freelamp.com article 0328, section "技术突破：极坐标量化": random
  orthogonal rotation first; no per-block scaling constants.
* [freelamp QJL]  same article, section "误差补偿：QJL 变换与 1-bit 残差修正":
  1-bit signs of the residual combined with the high-precision query give a
  zero-bias estimate.
* [csdn budget]   gitcode.csdn.net article, section "TurboQuant原理剖析": r kept
  at 16 bits, 2- or 3-bit codes, plus 1 QJL bit per dimension (3 or 4 bits in
  total).
* [csdn PolarQuant] same article, section "PolarQuant": rotate first; 4-D
  example where Q maps a column vector X to [5,5,5,5]^T.
* [csdn polar]    same article, section "将笛卡尔积坐标转为极坐标": r = ||x||_2,
  stored at higher precision (FP16).
* [csdn QJL-1/2/3] same article, section "QJL", steps 1 (residual = original
  minus PolarQuant reconstruction, then a Gaussian JL projection), 2 (keep only
  the signs: >0 -> 1, <0 -> 0) and 3 (the query against the signs gives an
  unbiased correction added to the PolarQuant result).
* [nonnda 3.4]    nonndazone.ru essay on TurboQuant and embedding geometry,
  section 3.4: one precomputed scheme (e.g. centroids) for all tokens and
  layers; section 3.2: centroids placed where probability is higher.
"""

from .rng import splitmix64_stream, gaussian_stream, haar_rotation, jl_matrix, method_matrices
from .codebook import Codebook, sphere_codebook, sphere_marginal_pdf, sphere_cell_prob, sphere_cell_first_moment
from .turboquant import (
    Quantized, quantize, dequantize, qjl_signs, pack_planes, unpack_planes, pack_signs,
    unpack_signs, estimate, estimate_all, attention_logits, attention_values, attention_output,
    search_topk, recall_at_1, fp16_round, QJL_CONST, SplitCodebook, split_quantize, split_dequantize,
    split_estimate, pack_split, unpack_split,
)
from . import paged
from .polar import (
    polar_forward, polar_inverse, angle_pdf, angle_cdf, angle_dof, AngleCodebook, angle_codebook,
    PolarCodebook, polar_codebook, PolarQuantized, polar_codes, polar_rebuild, polar_dequantize,
    polar_quantize, polar_estimate, polar_words, pack_polar, unpack_polar,
)

__all__ = [
    "paged",
    "polar_forward", "polar_inverse", "angle_pdf", "angle_cdf", "angle_dof", "AngleCodebook",
    "angle_codebook", "PolarCodebook", "polar_codebook", "PolarQuantized", "polar_codes",
    "polar_rebuild", "polar_dequantize", "polar_quantize", "polar_estimate", "polar_words",
    "pack_polar", "unpack_polar",
    "splitmix64_stream", "gaussian_stream", "haar_rotation", "jl_matrix", "method_matrices",
    "Codebook", "sphere_codebook", "sphere_marginal_pdf", "sphere_cell_prob",
    "sphere_cell_first_moment", "Quantized", "quantize", "dequantize", "qjl_signs",
    "pack_planes", "unpack_planes", "pack_signs", "unpack_signs", "estimate", "estimate_all",
    "attention_logits", "attention_values", "attention_output", "search_topk", "recall_at_1", "fp16_round",
    "SplitCodebook", "split_quantize", "split_dequantize", "split_estimate", "pack_split", "unpack_split",
    "QJL_CONST",
]
from . import sharded
