"""The library keeps no per-call state outside the caller's buffers and the
call's own stream-ordered workspace (the dQ kernel's work counter included),
so forward + backward steps of different shapes enqueued on two streams at
once give the same bits as the same steps run one after the other (dQ of the
D = 64 backward up to the order of its float32 sums)."""
import pytest
import torch

import online_softmax_05_gb300 as fa
from online_softmax_05_gb300.inputs import make_inputs
from tests.tolerances import same_gradients


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_softmax_05_gb300 import build
    build.build()
    fa.load_library()


CASES = [((2, 4, 1000, 128), True, 51), ((1, 8, 777, 64), False, 52), ((3, 2, 2048, 128), True, 53)]


def step(inputs, causal, stream):
    q, k, v, do = inputs
    o, lse = fa.attention_forward(q, k, v, causal=causal, stream=stream)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, causal=causal, stream=stream)
    return o, lse, dq, dk, dv


@pytest.mark.gpu
def test_two_streams_match_sequential():
    dev = torch.device("cuda")
    inputs = [tuple(t.to(dev) for t in make_inputs(*shape, seed=seed)) for shape, _, seed in CASES]
    ref = [step(x, causal, torch.cuda.current_stream(dev)) for x, (_, causal, _) in zip(inputs, CASES)]
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    streams = [torch.cuda.Stream(dev) for _ in CASES]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream(dev))
    got = []
    for rep in range(3):   # several rounds, so the calls on different streams overlap
        got = []
        for x, (_, causal, _), s in zip(inputs, CASES, streams):
            with torch.cuda.stream(s):
                got.append(step(x, causal, s))
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    for outs, want, (shape, _, _) in zip(got, ref, CASES):
        for a, b in zip(outs[:2], want[:2]):
            assert torch.equal(a, b)
        assert same_gradients(outs[2:], want[2:], shape[3])
