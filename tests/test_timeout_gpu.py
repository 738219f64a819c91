"""Failure detection without a GPU fault: a bounded device-side wait is made to
run out on purpose and must come back as a status code, leaving the context
usable.

The workspace header carries the wait limit (max_spin) and a test hook
(hold_item): when hold_item is set, the TMA producer of the tensor-core causal
path never issues its first load, so the consumers' waits on that load cannot
complete. Each wait gives up after max_spin microseconds, the kernel records
LA_ERR_TIMEOUT in the header and returns; la_query_status reports it.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import make_qkv, to_f64

pytestmark = pytest.mark.gpu

MAX_SPIN_WORD, HOLD_WORD = 4, 5   # uint32 index of max_spin and hold_item in the header


@pytest.fixture(scope="module")
def la():
    import linear_attention_elu_gb300 as m
    return m


def test_withheld_load_times_out_and_context_survives(la):
    dev = torch.device("cuda")
    q, k, v = make_qkv(2, 2, 1000, 64, "bf16", seed=3)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    ws = la.workspace(la.LA_OP_CAUSAL, 2, 2, 1000, 64, 64, torch.bfloat16, dev)
    hdr = ws[:256].view(torch.int32)
    hdr[MAX_SPIN_WORD] = 2000  # 2 ms
    hdr[HOLD_WORD] = 1
    la.la_causal_fwd(qd, kd, vd, ws=ws)
    assert la.la_query_status(ws) == la.LA_ERR_TIMEOUT
    assert la.la_query_status(ws) == 0          # the status word was cleared
    la.la_workspace_init(ws)                     # default limit, hook off
    o = la.la_causal_fwd(qd, kd, vd, ws=ws)
    assert la.la_query_status(ws) == 0
    ref = oracle.recurrent(to_f64(q), to_f64(k), to_f64(v), True)
    got = to_f64(o)
    err = (np.abs(got - ref).max(-1) / np.abs(ref).max(-1)).max()
    assert err <= 2e-2


@pytest.mark.parametrize("D", [64, 128])
def test_withheld_load_times_out_noncausal(la, D):
    dev = torch.device("cuda")
    q, k, v = make_qkv(1, 4, 700, D, "bf16", seed=4)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    ws = la.workspace(la.LA_OP_NONCAUSAL, 1, 4, 700, D, D, torch.bfloat16, dev)
    hdr = ws[:256].view(torch.int32)
    hdr[MAX_SPIN_WORD] = 2000  # 2 ms
    hdr[HOLD_WORD] = 1
    la.la_noncausal_fwd(qd, kd, vd, ws=ws)
    assert la.la_query_status(ws) == la.LA_ERR_TIMEOUT
    la.la_workspace_init(ws)
    o = la.la_noncausal_fwd(qd, kd, vd, ws=ws)
    assert la.la_query_status(ws) == 0
    ref = oracle.recurrent(to_f64(q), to_f64(k), to_f64(v), False)
    got = to_f64(o)
    assert (np.abs(got - ref).max(-1) / np.abs(ref).max(-1)).max() <= 2e-2
