"""Stream ordering of calls whose second kernel (the log-sum-exp merge) is
launched early, with programmatic stream serialisation: attention with a split
last wave and the split-KV decode, enqueued back to back on one stream with no
synchronisation in between, must give exactly the results of the same calls
made one at a time."""
import pytest
import torch

from cascaded_reductions_pass_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_attention_split_tail_back_to_back(rf):
    n = 10
    cases = [tuple(t.cuda() for t in inputs.attn_inputs(1, 8, 8, 1024, 1024, 64, "f16", seed=200 + i))
             for i in range(n)]
    ws = rf.attn_workspace(*cases[0][:2])
    assert ws is not None, "the shape must exercise the split tail"
    solo = []
    for q, k, v in cases:
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
        rf.rf_attn_fwd_ex(q, k, v, o, lse, scale=0.125, workspace=ws)
        torch.cuda.synchronize()
        solo.append((o, lse))
    outs = [(torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")) for q, _, _ in cases]
    for (q, k, v), (o, lse) in zip(cases, outs):  # one workspace, reused by every call in stream order
        rf.rf_attn_fwd_ex(q, k, v, o, lse, scale=0.125, workspace=ws)
    torch.cuda.synchronize()
    for (o, lse), (o1, lse1) in zip(outs, solo):
        assert torch.equal(o, o1) and torch.equal(lse, lse1)


def test_decode_back_to_back(rf):
    n = 10
    B, Hq, Hkv, L, D, S = 2, 16, 2, 4096, 128, 8
    cases = [tuple(t.cuda() for t in inputs.decode_inputs(B, Hq, Hkv, L, D, "bf16", seed=300 + i)) for i in range(n)]
    ws = rf.decode_workspace(B, Hq, D, S)
    solo = []
    for q, kc, vc in cases:
        o, lse = rf.decode(q, kc, vc, S, workspace=ws)
        torch.cuda.synchronize()
        solo.append((o, lse))
    outs = [rf.decode(q, kc, vc, S, workspace=ws) for q, kc, vc in cases]
    torch.cuda.synchronize()
    for (o, lse), (o1, lse1) in zip(outs, solo):
        assert torch.equal(o, o1) and torch.equal(lse, lse1)
