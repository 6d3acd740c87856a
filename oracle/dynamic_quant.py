"""Oracle for DynamicQuant of q^N (per-row symmetric int8 quantisation).

Test infrastructure only (see oracle/__init__.py). Written from the page
"aclnnMlaPrologV3WeightNz" ("Formula", Dequant Scale Query Nope):
dequantScaleQNope = RowMax(abs(q^N)) / 127 and q^N = round(q^N /
dequantScaleQNope), with the scale of shape (T, N, 1) ("Shape restrictions"),
i.e. one scale per token and head, the row being the last axis (Hckv).

Everything is float64 and each result is rounded once:

* the quotient q / (RowMax/127) is the rational number q*127/RowMax. For
  inputs of at most 24 significant bits (every 16-bit or float32 value),
  q*127 is exact in float64 and one float64 division gives the correctly
  rounded quotient; an exact half-integer quotient stays exact, and a
  quotient that is not one lies far more than a float64 rounding error
  away from any half-integer, so the integer decided below is that of the
  exact rational;
* the code is round(quotient), round being round-half-to-even (the pages
  state their formulas in PyTorch terms; torch.round ties to even),
  clamped to [-127, 127] (only reachable through rounding error: the exact
  quotient of the row maximum is +-127);
* the returned scale is RowMax/127 rounded once to float32 (the type of
  dequantScaleQNope): the float64 quotient is not exact, but RowMax/127 has
  a binary expansion that repeats with period 7 (2^7 = 1 mod 127), so its
  float64 rounding never lands on a float32 rounding midpoint and the cast
  gives the correctly rounded float32 value;
* an all-zero row has scale 0 and codes 0 (the formula would divide 0 by 0).
"""
import numpy as np


def dynamic_quant_quotients(q):
    """q: float64 [rows, H] of 16-bit or float32 input values. Returns
    (v, rowmax): v[r, c] = q[r, c] / (rowmax[r] / 127) in float64 (0 on an
    all-zero row), before rounding to codes."""
    q = np.asarray(q, dtype=np.float64)
    rowmax = np.max(np.abs(q), axis=-1)
    safe = np.where(rowmax > 0, rowmax, 1.0)
    v = (q * 127.0) / safe[:, None]
    return v, rowmax


def ref_dynamic_quant(q):
    """q: float64 [rows, H] holding 16-bit input values. Returns
    (codes int8 [rows, H], scale float32 [rows])."""
    v, rowmax = dynamic_quant_quotients(q)
    codes = np.clip(np.rint(v), -127, 127).astype(np.int8)
    scale = (rowmax / 127.0).astype(np.float32)
    return codes, scale
