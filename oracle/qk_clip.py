"""fp64 CPU oracle of the QK-Clip rescale applied after the optimizer update.

TEST INFRASTRUCTURE ONLY; the product path never imports it.

Sources (page title, section):
  [KIMI] kimi-k3, "Optimization", "QK-Clip watches a different failure mode":
         per head, the maximum causally valid query-key score (scaled by the
         square root of the query-key dimension) is compared with a positive
         threshold tau; a head above it has selected unshared query and key
         projection rows rescaled after a successful optimizer update, with a
         factor below one distributed across the projection paths; a head
         below it gets gamma = 1; shared key and value projections stay.
  [DEW]  dew.training.optim, "scale_by_qk_clip" (tau = 100 by default; Kimi
         K2's MuonClip, applied after the update) and "QK_PROJECTIONS"
         (q_proj, q_b_proj, k_proj, kv_b_proj).

Readings (the page's formula for gamma is lost in extraction):
  * gamma_h = min(1, tau / s_h).
  * A rescale entry names a weight stored (rows, cols) with one block of
    head_stride rows per head; inside each block, scaled_rows rows starting
    at row_offset are multiplied by gamma_h ** exponent. Query and key rows
    of a head take exponents that sum to 1 (0.5 each by default), so the
    head's logits scale by exactly gamma_h; a query path whose key is shared
    (MLA's rotary part) takes exponent 1 and the shared key none.
  * Nothing is rescaled after a skipped step.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class ClipEntry:
    heads: int
    head_stride: int
    row_offset: int
    scaled_rows: int
    head_index0: int
    exponent: float = 0.5


def gamma(s_max, tau: float) -> np.ndarray:
    s = np.asarray(s_max, dtype=np.float64)
    return np.where(s > tau, tau / np.where(s > 0, s, 1.0), 1.0)


def qk_clip(W, entry: ClipEntry, s_max, tau: float, skipped: bool = False) -> np.ndarray:
    """The weight after [KIMI]'s rescale of one entry's rows."""
    W = np.array(W, dtype=np.float64, copy=True)
    if skipped:
        return W
    g = gamma(s_max, tau)
    for h in range(entry.heads):
        f = g[entry.head_index0 + h] ** entry.exponent
        r0 = h * entry.head_stride + entry.row_offset
        W[r0:r0 + entry.scaled_rows] *= f
    return W
