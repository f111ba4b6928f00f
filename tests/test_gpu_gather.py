"""quads_moe_gather called directly with hand-made expert offsets: rows copied
bit for bit into expert order, padding rows zero, and nothing written past
offsets[E] -- including a last 128-row block that the offsets end inside,
where the scale atoms are written a 4-byte group at a time.  Wide rows (2048
columns) and the narrow residual slices (64 and 256 columns) take different
code paths in the kernel."""
import numpy as np
import pytest
import torch

from helpers import unswizzle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cols", [64, 256, 2048])
@pytest.mark.parametrize("ends", [[0, 100, 250, 300], [0, 128, 128, 384], [0, 0, 0, 0], [0, 37, 37, 129]])
def test_gather_rows_into_expert_order(lib, cols, ends):
    from nvfp4_w4a4_quantized_quant_gb300 import quads as Q
    dev = torch.device("cuda", 0)
    T, cap = 200, 512
    g = torch.Generator().manual_seed(cols * 7 + ends[-1])
    x = (torch.randn(T, cols, generator=g) * 3).to(torch.bfloat16).to(dev)
    q, _ = Q.quantize_nvfp4(x)
    nr = ends[-1]
    row_token = torch.randint(-1, T, (cap,), generator=g, dtype=torch.int32)
    plan = dict(row_token=row_token.to(dev), offsets=torch.tensor(ends, dtype=torch.int32, device=dev),
                experts=len(ends) - 1, rows_capacity=cap)
    oc = torch.full((cap, cols // 2), 0xAB, dtype=torch.uint8, device=dev)
    osf = torch.full((Q.sf_tc_bytes(cap, cols),), 0xCD, dtype=torch.uint8, device=dev)
    out = Q.moe_gather(plan, q, out=(oc, osf))
    torch.cuda.synchronize()
    assert out.codes.data_ptr() == oc.data_ptr()

    ic, isf = q.codes.cpu().numpy(), q.scales.cpu().numpy().reshape(T, cols // 16)
    rt = row_token.numpy()[:nr]
    want_c = np.where(rt[:, None] >= 0, ic[np.maximum(rt, 0)], 0).astype(np.uint8)
    want_s = np.where(rt[:, None] >= 0, isf[np.maximum(rt, 0)], 0).astype(np.uint8)
    got_c = oc.cpu().numpy()
    got_s = unswizzle(osf, cap, cols)
    assert np.array_equal(got_c[:nr], want_c)
    assert np.array_equal(got_s[:nr], want_s)
    assert (got_c[nr:] == 0xAB).all()        # rows past offsets[E] untouched
    assert (got_s[nr:] == 0xCD).all()
