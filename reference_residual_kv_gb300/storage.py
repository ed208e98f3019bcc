"""Storage accounting for the compressed cache (host arithmetic only).

Two views are kept apart:

* the ResidualKV paper's keep ratio (KR) formula, reading notes §3.3 (paper
  Sec. V-A): with beta = H_full / H the share of full-attention layers,
      q_b = b/16 + 2/32                      (b-bit payload + two FP16 extremes per 32)
      KR  = beta q_4 + (1 - beta)(rho_ref / 2 + q_b d_c / (2 d_k));
* the bytes this library actually stores per token (fp32 group extremes, so that a
  constant group is kept exactly, and the per-token reference relation, which the
  paper's KR leaves out).
"""
from __future__ import annotations


def q_b(bits: int, group: int = 32, extreme_bits: int = 16) -> float:
    """Relative size of a b-bit grouped code vs FP16: payload plus two extremes per group."""
    return bits / 16.0 + 2.0 * extreme_bits / (16.0 * group)


def paper_keep_ratio(beta: float, rho_ref: float, dc_over_2dk: float, bits: int,
                     full_bits: int = 4) -> float:
    """KR of the paper: full layers at q_{full_bits}, sparse layers FP8 references
    (half of FP16) at density rho_ref plus b-bit residual codes of width d_c."""
    return beta * q_b(full_bits) + (1.0 - beta) * (0.5 * rho_ref + q_b(bits) * dc_over_2dk)


def record_bytes(d_c: int, bits: int, group: int = 32, k: int = 4) -> int:
    """Bytes of one non-reference token's record in this library's layout:
    packed codes, {z_min, delta} as two fp32 per group, k int32 reference slots."""
    n_groups = (d_c + group - 1) // group
    return d_c * bits // 8 + 8 * n_groups + 4 * k


def layer_bytes_per_token(W: int, d_c: int, bits: int, stride: int, ref_elem_bytes: int,
                          group: int = 32, k: int = 4) -> float:
    """Average stored bytes per token of one layer-sequence: every token keeps a record
    (a reference's record is all zero but present, which keeps random access uniform),
    and one token in `stride` also keeps its reference vector."""
    return record_bytes(d_c, bits, group, k) + W * ref_elem_bytes / stride
