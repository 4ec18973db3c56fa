"""VMM-backed output workspace: a reserved virtual range whose physical pages are bound only as
the chunk output grows (the Global Memory Manager idea at the scale of this operator)."""
import pytest
import torch

from masked_token_lm_gb300 import mosaic as mz
from masked_token_lm_gb300 import workloads as wl
from oracle import mask_only_logits as orc
from tests.parity_utils import assert_close, bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def test_workspace_binds_on_demand_with_a_stable_address():
    ws = mz.Workspace(64 << 30)  # 64 GiB of address space, no memory yet
    try:
        assert ws.reserved_bytes >= 64 << 30 and ws.bound_bytes == 0
        p1 = ws.bind(100 << 20)
        assert ws.bound_bytes >= 100 << 20
        small = ws.tensor((1000, 1000), torch.float32)
        small.fill_(3.0)
        p2 = ws.bind(1 << 30)  # grow: same base address, earlier contents kept
        assert p2 == p1 and ws.bound_bytes >= 1 << 30
        assert float(small.sum()) == 3.0 * 1000 * 1000
        ws.trim(0)
        assert ws.bound_bytes == 0
        p3 = ws.bind(4 << 20)
        assert p3 == p1
        with pytest.raises(mz.MosaicError) as e:
            ws.bind(65 << 30)
        assert e.value.status == mz.MOSAIC_ERR_UNSUPPORTED
    finally:
        ws.close()


def test_workspace_as_lazy_chunk_output_matches_plain_buffer():
    L, d, V, M = 3000, 512, 4104, 900
    H, W = wl.make_hidden(L, d, 61, DEV), wl.make_weight(V, d, 62, DEV)
    idx = wl.uniform_positions(L, M, seed=63).to(DEV)
    mo = mz.Mosaic(0)
    ref = mo.masked_logits(H, idx, W, out_dtype=torch.bfloat16)
    assert mo.check() == mz.MOSAIC_OK
    # the plain-buffer result itself against the oracle (fp64), every element
    exact = orc.masked_logits(bits(H), idx.cpu().numpy(), bits(W))
    assert_close(ref, exact, torch.bfloat16, "plain buffer vs oracle")
    ws = mz.Workspace(M * V * 2)  # reserved for the unchunked output, bound per chunk size
    try:
        full = torch.empty((M, V), dtype=torch.bfloat16, device=DEV)
        for chunk_rows in (128, 300):
            out = ws.tensor((chunk_rows, V), torch.bfloat16)
            assert ws.bound_bytes < M * V * 2

            def on_chunk(c, rb, rows, buf):
                full[rb:rb + rows].copy_(buf[:rows])

            mo.masked_logits(H, idx, W, out=out, chunk_rows=chunk_rows, on_chunk=on_chunk)
            assert mo.check() == mz.MOSAIC_OK
            assert torch.equal(full.view(torch.int16), ref.view(torch.int16))
            assert_close(full, exact, torch.bfloat16, f"workspace chunks of {chunk_rows} vs oracle")
    finally:
        torch.cuda.synchronize()
        del out
        ws.close()
        mo.close()
