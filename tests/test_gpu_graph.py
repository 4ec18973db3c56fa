"""The public calls captured into a CUDA graph (as bench.py times them) and replayed give the
direct call's results bit for bit: logits (unchunked and chunked, flat and CSR), the E4M3 path
with its per-call quantization of the masked hidden rows, and fused sampling."""
import pytest
import torch

from masked_token_lm_gb300 import mosaic as mz
from masked_token_lm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def mo():
    m = mz.Mosaic(0)
    yield m
    m.close()


def capture(fn):
    """fn(stream) enqueues the work; returns a graph holding it (captured on a side stream)."""
    s = torch.cuda.Stream(device=DEV)
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
        fn(s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("csr,chunk_rows", [(False, 0), (False, 100), (True, 0), (True, 64)])
def test_graph_replay_of_masked_logits_is_bitwise_the_direct_call(mo, csr, chunk_rows):
    d, V = 256, 1032
    if csr:
        m = wl.ragged_mask(4, 300, seed=5).to(DEV)
        L = int(m.seq_offsets[-1])
        idx, so, moff = m.idx, m.seq_offsets, m.mask_offsets
    else:
        L = 1200
        idx, so, moff = wl.uniform_positions(L, 300, seed=6).to(DEV), None, None
    H, W = wl.make_hidden(L, d, 7, DEV), wl.make_weight(V, d, 8, DEV)
    M = int(idx.numel())
    direct = mo.masked_logits(H, idx, W, so, moff)
    rows_out = chunk_rows if 0 < chunk_rows < M else M
    out = torch.empty((rows_out, V), dtype=torch.bfloat16, device=DEV)
    full = torch.zeros((M, V), dtype=torch.bfloat16, device=DEV)

    def on_chunk(c, rb, rows, buf):  # runs at capture time; the copy it enqueues is captured
        full[rb:rb + rows].copy_(buf[:rows])

    before = mo.launches
    g = capture(lambda s: mo.masked_logits(H, idx, W, so, moff, out=out, chunk_rows=chunk_rows,
                                           on_chunk=on_chunk if rows_out < M else None, stream=s))
    captured = mo.launches - before
    assert captured == -(-M // rows_out)
    for _ in range(2):
        full.zero_()
        g.replay()
        torch.cuda.synchronize()
        got = full if rows_out < M else out
        assert torch.equal(got.view(torch.int16), direct.view(torch.int16))
    assert mo.launches - before == captured  # replays enqueue nothing through the host
    assert mo.check() == mz.MOSAIC_OK


def test_graph_replay_of_fp8_step_is_bitwise_the_direct_call(mo):
    L, d, V, M = 900, 256, 776, 300
    H, W = wl.make_hidden(L, d, 11, DEV), wl.make_weight(V, d, 12, DEV)
    idx = wl.uniform_positions(L, M, seed=13).to(DEV)
    qW, sW = mz.quantize_rows_e4m3(W)
    qH = torch.zeros((L, d), dtype=torch.uint8, device=DEV)
    sH = torch.zeros(L, dtype=torch.float32, device=DEV)
    mz.quantize_masked_rows_e4m3(H, idx, qH, sH)
    direct = mo.masked_logits_fp8(qH, sH, idx, qW, sW)
    qH.zero_()
    sH.zero_()
    out = torch.empty_like(direct)

    def step(s):
        mz.quantize_masked_rows_e4m3(H, idx, qH, sH, stream=s)
        mo.masked_logits_fp8(qH, sH, idx, qW, sW, out=out, stream=s)

    g = capture(step)
    H.mul_(2.0)  # the replay must read the hidden states as they are at replay time
    g.replay()
    torch.cuda.synchronize()
    direct2 = mo.masked_logits_fp8(*mz.quantize_rows_e4m3(H), idx, qW, sW)
    assert torch.equal(out.view(torch.int16), direct2.view(torch.int16))
    H.mul_(0.5)  # exact: back to the original values
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), direct.view(torch.int16))
    assert mo.check() == mz.MOSAIC_OK


def test_graph_replay_of_masked_sample_matches_the_direct_call(mo):
    L, d, V, M = 1000, 256, 1032, 300
    H, W = wl.make_hidden(L, d, 21, DEV), wl.make_weight(V, d, 22, DEV)
    idx = wl.uniform_positions(L, M, seed=23).to(DEV)
    tok, conf = mo.masked_sample(H, idx, W)
    ws = torch.empty(mz.mosaic_masked_sample_workspace_bytes(M, V), dtype=torch.uint8, device=DEV)
    res = {}
    g = capture(lambda s: res.update(zip(("tok", "conf"),
                                         mo.masked_sample(H, idx, W, workspace=ws, stream=s))))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(res["tok"], tok)
    assert torch.equal(res["conf"].view(torch.int32), conf.view(torch.int32))
    assert mo.check() == mz.MOSAIC_OK
