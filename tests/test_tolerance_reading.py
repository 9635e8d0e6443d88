"""Why the O bound allows the bf16 output's own rounding (host only).

The pages' forward rounds the probabilities to bf16 before P V ("Triton
FlashAttention-2 forward", "The kernel": the dot product takes
p.to(v.dtype)) while the row sum l is accumulated from the unrounded P, and
the result is returned in bf16.  Replaying that recurrence in float64 on one
row of the large-logit workload (B=8 H=32 T=3000 D=128, Q and K ~ N(0, 4^2),
batch 0, head 26, row 1544; its two heaviest keys weigh 0.53 and 0.40) shows
the two parts of the error separately: before the final rounding the
recurrence is within 1e-2 of the exact O; the rounding to bf16 (spacing 2^-6
near 2.08) then takes one element past 1e-2, but not past 1e-2 plus half a
bf16 ulp.  That is the bound tests/tolerances.py states."""
import numpy as np
import torch

import oracle
from online_softmax_05_gb300.inputs import WORKLOADS, workload_inputs, to_f64
from tests.tolerances import O_TOL, bf16_half_ulp, o_bound


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.bfloat16).to(torch.float64).numpy()


def _recurrence_with_bf16_p(q_row, k, v, scale, bn):
    """"Lab 06", section 3 recurrence for one query row, key tiles of bn,
    with P rounded to bf16 before it multiplies V (float64 elsewhere)."""
    s = (k @ q_row) * scale
    m, l, acc = -np.inf, 0.0, np.zeros(v.shape[1])
    for j0 in range(0, k.shape[0], bn):
        sj = s[j0:j0 + bn]
        m_new = max(m, sj.max())
        alpha = np.exp(m - m_new)
        p = np.exp(sj - m_new)
        l = alpha * l + p.sum()
        acc = alpha * acc + _bf16(p) @ v[j0:j0 + bn]
        m = m_new
    return acc / l


def test_output_rounding_is_what_crosses_1e2():
    w = WORKLOADS["ragged_b8h32t3000d128"]
    q, k, v, _ = workload_inputs(w)
    b, h, row = 0, 26, 1544
    qf, kf, vf = (to_f64(t[b, h]) for t in (q, k, v))
    o_ref = oracle.attn_fwd_rows(qf, kf, vf, w.scale, False, [row])[0][0]
    for bn in (64, 128):
        o = _recurrence_with_bf16_p(qf[row], kf, vf, w.scale, bn)
        before = np.abs(o - o_ref)
        after = np.abs(_bf16(o) - o_ref)
        assert before.max() <= O_TOL / 2            # the recurrence itself is well inside 1e-2
        assert after.max() > O_TOL                  # the bf16 output rounding crosses it
        assert np.all(after <= o_bound(o_ref))      # and stays inside 1e-2 + half an ulp
        assert after.max() - before.max() <= bf16_half_ulp(o_ref).max()
