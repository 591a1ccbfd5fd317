"""GPU parity of the integer / byte steps: the schedule and the MXFP8 quantiser
must match the oracle bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_mok_gb300 import inputs as gen
from tests.gpu_util import mok

pytestmark = pytest.mark.gpu


def _check_schedule(te, E, c):
    m = mok()
    s = m.schedule(te.cuda(), E, c)
    st, nt, P = s.status()
    ref = oracle.build_schedule(te.numpy(), E, c)
    assert st == ref["status"] == 0
    assert nt == ref["num_tiles"] and P == ref["P"]
    arr = {k: v.cpu().numpy() for k, v in s.arrays().items()}
    for key in ("cnt", "row0", "row_src", "slot_row", "tile_expert", "tile_row0", "tile_rows"):
        assert np.array_equal(arr[key], ref[key]), key
    assert arr["header"][3] == ref["num_primary"]
    _check_pairs(arr, ref)
    _check_groups(arr, ref)


def _check_pairs(arr, ref):
    """The tile pairs of the CTA-pair GEMMs: consecutive tiles of one expert,
    paired from the start of its run within the primary list, then within the
    overflow list; each tile in exactly one pair."""
    nt, npr = ref["num_tiles"], ref["num_primary"]
    te = ref["tile_expert"]
    want = []
    for lo, hi in ((0, npr), (npr, nt)):
        i = lo
        while i < hi:
            j = i + 1 if i + 1 < hi and te[i + 1] == te[i] else -1
            want.append((i, j))
            i += 2 if j >= 0 else 1
    pairs = arr["pair_tile"].reshape(-1, 2)
    assert arr["header"][4] == len(want)
    assert [tuple(int(v) for v in p) for p in pairs[:len(want)]] == want
    assert np.all(pairs[len(want):] == -1)


def _run_groups(experts, lo, hi, cap):
    """Work-group entries of units [lo, hi): each run of one expert cut evenly
    into groups of at most cap units; entry = position | length << 8."""
    want, i = {}, lo
    while i < hi:
        j = i
        while j < hi and experts[j] == experts[i]:
            j += 1
        n = j - i
        ng = -(-n // cap)
        size = -(-n // ng)
        for q in range(n):
            start = q // size * size
            want[i + q] = (q - start) | (min(size, n - start) << 8)
        i = j
    return want


def _check_groups(arr, ref):
    """The GEMMs' work groups (unit_group): runs of one expert's tiles within
    the primary and the overflow list, and of its pairs, cut evenly into groups
    of at most 32 tiles or 16 pairs; unused entries -1."""
    nt, npr, mt = ref["num_tiles"], ref["num_primary"], len(ref["tile_expert"])
    te = ref["tile_expert"]
    g = arr["unit_group"]
    want = {**_run_groups(te, 0, npr, 32), **_run_groups(te, npr, nt, 32)}
    assert [int(g[t]) for t in range(nt)] == [want[t] for t in range(nt)]
    assert np.all(g[nt:mt] == -1)
    pairs = arr["pair_tile"].reshape(-1, 2)
    npairs = int(arr["header"][4])
    pe = [te[pairs[p][0]] for p in range(npairs)]
    prim_pairs = sum(1 for p in range(npairs) if pairs[p][0] < npr)
    want = {**_run_groups(pe, 0, prim_pairs, 16), **_run_groups(pe, prim_pairs, npairs, 16)}
    assert [int(g[mt + p]) for p in range(npairs)] == [want[p] for p in range(npairs)]
    assert np.all(g[mt + npairs:] == -1)


@pytest.mark.parametrize("T,k,E,skew,c", [
    (128, 2, 8, None, 0.5),            # tiny layer
    (4096, 8, 64, None, 0.5),          # bf16 / mxfp8 T=4096 layers
    (16384, 8, 128, 1.2, 0.5),         # skewed routing, capacity 0.5
    (16384, 8, 128, 1.2, 1.0),         # skewed routing, capacity 1.0
    (65536, 8, 256, None, 0.5),        # large layer
    (1, 1, 1, None, 0.5), (5, 3, 7, None, 0.0), (4097, 5, 1000, None, 0.5), (3000, 16, 64, 1.2, 0.01),
    (8192, 8, 64, 1.2, 0.5), (65537, 1, 16, 1.2, 0.5),
    # multipliers that float32 cannot hold, where c*T lands on a whole tile in
    # double precision but just above it in float32 (the tile order differs)
    (2560, 8, 16, 1.2, 0.05), (1280, 8, 16, 1.2, 0.1), (1280, 4, 32, 1.2, 0.3), (640, 8, 16, 1.2, 0.6),
])
def test_schedule_bit_exact(T, k, E, skew, c):
    te = gen.make_routing(T, k, E, seed=T + E, skew=skew)
    _check_schedule(te, E, c)


def test_schedule_repeated_calls_identical():
    m = mok()
    te = gen.make_routing(8192, 8, 64, seed=3).cuda()
    a = m.schedule(te, 64, 0.5)
    b = m.schedule(te, 64, 0.5)
    torch.cuda.synchronize()
    for (name, x), y in zip(a.arrays().items(), b.arrays().values()):
        assert torch.equal(x, y), name


def test_schedule_bad_expert_id_reports_index_error():
    m = mok()
    te = gen.make_routing(300, 4, 16, seed=1)
    te[123, 2] = 16
    s = m.schedule(te.cuda(), 16, 0.5)
    st, nt, P = s.status()
    assert st == 2 and nt == 0
    te[123, 2] = -5
    assert m.schedule(te.cuda(), 16, 0.5).status()[0] == 2


def _check_quant(x):
    m = mok()
    codes, scales = m.mxfp8_quantize(x.cuda())
    rc, rs = oracle.mxfp8_quantize(x.double().reshape(-1, x.shape[-1]).numpy())
    assert np.array_equal(codes.cpu().numpy().reshape(rc.shape), rc)
    assert np.array_equal(scales.cpu().numpy().reshape(rs.shape), rs)


@pytest.mark.parametrize("R,K,std", [(1, 32, 1.0), (257, 96, 1.0), (1024, 2048, 0.02), (64, 7168, 3.0),
                                     (2048, 4096, 1e-3)])
def test_quantize_bit_exact(R, K, std):
    _check_quant(gen.make_matrix(R, K, std=std, seed=R + K))


def test_quantize_edge_values():
    table = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    fin = table[np.isfinite(table)]
    # exact grid values and midpoints scaled by assorted powers of two, zeros,
    # negative zeros, tiny and huge magnitudes, bf16 subnormals
    mids = (np.sort(np.unique(np.abs(fin)))[1:] + np.sort(np.unique(np.abs(fin)))[:-1]) / 2
    v = np.concatenate([fin, mids, -mids, [0.0, -0.0] * 16, [3e38, -3e38, 1e-38, -1e-39, 9e-41, -9e-41]])
    v = np.concatenate([v * 2.0 ** s for s in (-100, -9, 0, 3, 100)])
    x = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
    x = x[torch.isfinite(x)]           # the quantiser's inputs are finite
    x = x[: x.numel() // 32 * 32].reshape(-1, 32)
    _check_quant(x)
    # all-zero and single-nonzero blocks
    z = torch.zeros(4, 64, dtype=torch.bfloat16)
    z[1, 5] = -1.0
    z[2, 40] = 448.0
    z[3, :] = -0.0
    _check_quant(z)


def test_quantize_empty():
    m = mok()
    c, s = m.mxfp8_quantize(torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"))
    assert c.numel() == 0 and s.numel() == 0


def _check_quant_t(x3):
    """The transposing quantiser against the oracle's quantiser applied to the
    transpose of each matrix of the batch, bit for bit; the dual quantiser
    gives that and the row-wise quantisation from one read."""
    m = mok()
    codes, scales = m.mxfp8_quantize_t(x3.cuda())
    (dc, ds), (dtc, dts) = m.mxfp8_quantize_dual(x3.cuda())
    for b in range(x3.shape[0]):
        rc, rs = oracle.mxfp8_quantize(x3[b].double().numpy().T)
        assert np.array_equal(codes[b].cpu().numpy(), rc), b
        assert np.array_equal(scales[b].cpu().numpy(), rs), b
        assert np.array_equal(dtc[b].cpu().numpy(), rc), b
        assert np.array_equal(dts[b].cpu().numpy(), rs), b
        qc, qs = oracle.mxfp8_quantize(x3[b].double().numpy())
        assert np.array_equal(dc[b].cpu().numpy(), qc), b
        assert np.array_equal(ds[b].cpu().numpy(), qs), b


@pytest.mark.parametrize("B,R,C,std", [(1, 32, 64, 1.0), (3, 160, 192, 0.02), (2, 1024, 2048, 0.02),
                                       (1, 2048, 64, 3.0), (4, 128, 128, 1e-3)])
def test_quantize_t_bit_exact(B, R, C, std):
    x = gen.make_matrix(B * R, C, std=std, seed=B + R + C).reshape(B, R, C).contiguous()
    _check_quant_t(x)


def test_quantize_t_edge_values():
    table = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    fin = table[np.isfinite(table)]
    mids = (np.sort(np.unique(np.abs(fin)))[1:] + np.sort(np.unique(np.abs(fin)))[:-1]) / 2
    v = np.concatenate([fin, mids, -mids, [0.0, -0.0] * 16, [3e38, -3e38, 1e-38, -1e-39]])
    v = np.concatenate([v * 2.0 ** s for s in (-100, -9, 0, 3, 100)])
    x = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
    x = x[torch.isfinite(x)]
    n = x.numel() // (32 * 64) * (32 * 64)
    x = x[:n].reshape(-1, 32, 64).permute(1, 0, 2).reshape(32, -1)   # 32-row blocks of mixed values
    x = x[:, : x.shape[1] // 64 * 64].contiguous()
    z = torch.zeros(64, 64, dtype=torch.bfloat16)                    # zero and single-value blocks
    z[5, 1] = -1.0
    z[40, 2] = 448.0
    z[:, 3] = -0.0
    _check_quant_t(x.unsqueeze(0))
    _check_quant_t(z.unsqueeze(0))
    m = mok()
    c2, s2 = m.mxfp8_quantize_t(z.cuda())                            # a single matrix
    assert c2.shape == (64, 64) and s2.shape == (64, 2)
