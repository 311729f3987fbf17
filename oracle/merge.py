"""Oracle: merge of (O, m, l) partials from KV shards. Test infrastructure only.

6D attention notes §2.1, step 3 of the ring loop: after each step's local attention
the running state is updated with the step's partial -- the new maximum is the
larger of the two maxima, each side is rescaled by the exponential of its old
maximum minus the new one (alpha for the accumulator, beta for the step), the
row sums and the unnormalised outputs are combined with those weights, and the
loop ends by dividing the output by the row sum.

This module runs that fold in the pages' order (shard 0 first). fp64 throughout.

Reading where the pages are silent: a partial with no admissible key (m = -inf or
l = 0) contributes nothing; the fold would otherwise evaluate exp(-inf - (-inf)).
If every partial of a row is empty the row's output is 0 and its LSE is -inf.
"""

import numpy as np


def merge_partials(o_parts, m_parts, l_parts):
    """Fold n shard partials.

    o_parts [n, rows, d], m_parts [n, rows], l_parts [n, rows] (natural-log units).
    Returns (o [rows, d], lse [rows]) in fp64.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    m_parts = np.asarray(m_parts, dtype=np.float64)
    l_parts = np.asarray(l_parts, dtype=np.float64)
    n, rows, d = o_parts.shape
    o_acc = np.zeros((rows, d))
    m_acc = np.full(rows, -np.inf)
    l_acc = np.zeros(rows)
    for step in range(n):
        o_step, m_step, l_step = o_parts[step], m_parts[step], l_parts[step]
        empty_step = ~np.isfinite(m_step) | (l_step == 0)
        m_step = np.where(empty_step, -np.inf, m_step)
        m_new = np.maximum(m_acc, m_step)
        acc_live = np.isfinite(m_acc)
        step_live = np.isfinite(m_step)
        with np.errstate(invalid="ignore"):  # -inf - (-inf) is masked out below
            alpha = np.where(acc_live, np.exp(np.where(acc_live, m_acc - m_new, 0.0)), 0.0)
            beta = np.where(step_live, np.exp(np.where(step_live, m_step - m_new, 0.0)), 0.0)
        l_acc = alpha * l_acc + beta * np.where(step_live, l_step, 0.0)
        o_acc = alpha[:, None] * o_acc + beta[:, None] * np.where(step_live[:, None], o_step, 0.0)
        m_acc = m_new
    live = l_acc > 0
    safe_l = np.where(live, l_acc, 1.0)
    o = np.where(live[:, None], o_acc / safe_l[:, None], 0.0)
    lse = np.where(live, m_acc + np.log(safe_l), -np.inf)
    return o, lse
