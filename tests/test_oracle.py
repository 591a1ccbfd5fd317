"""Pins for the CPU oracle: each check ties the oracle to something other than
itself (published format tables, brute force, library routines, closed forms,
finite differences, invariants)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from mixture_experts_layer_mok_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pairs(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------ schedule

def _brute_schedule(te, E):
    T, k = te.shape
    flat = te.reshape(-1)
    order = sorted(range(T * k), key=lambda f: (flat[f], f))
    return order


@pytest.mark.parametrize("T,k,E,skew,seed", [
    (128, 2, 8, None, 0), (37, 3, 5, None, 1), (300, 8, 64, 1.2, 2),
    (1, 1, 1, None, 3), (129, 1, 1, None, 4), (64, 4, 200, None, 5)])
def test_schedule_matches_brute_force(T, k, E, skew, seed):
    te = gen.make_routing(T, k, E, seed=seed, skew=skew).numpy()
    s = O.build_schedule(te, E)
    assert s["status"] == 0
    flat = te.reshape(-1)
    order = _brute_schedule(te, E)
    # the non-padding rows, read in schedule order, are the brute-force order
    rs = s["row_src"][: s["P"]]
    assert list(rs[rs >= 0]) == order
    # invariants
    cnt = np.bincount(flat, minlength=E)
    assert (s["cnt"] == cnt).all() and s["cnt"].sum() == T * k
    padded = (cnt + 127) // 128 * 128
    assert (np.diff(s["row0"]) == padded).all() and s["row0"][0] == 0
    assert s["P"] == padded.sum() <= O.max_tiles(T, k, E) * 128
    f = np.arange(T * k)
    assert (s["row_src"][s["slot_row"]] == f).all()          # slot_row o row_src = id
    for e in range(E):                                         # rows of e stay in e's range
        lo, hi = s["row0"][e], s["row0"][e + 1]
        assert (flat[s["row_src"][lo:lo + cnt[e]]] == e).all()
        assert (s["row_src"][lo + cnt[e]:hi] == -1).all()
    assert (s["row_src"][s["P"]:] == -1).all()
    nt = s["num_tiles"]
    assert nt == ((cnt + 127) // 128).sum()
    assert (s["tile_rows"][:nt] >= 1).all() and (s["tile_rows"][:nt] <= 128).all()
    assert s["tile_rows"][:nt].sum() == T * k
    assert (s["tile_expert"][nt:] == -1).all()


def test_schedule_capacity_changes_order_only():
    te = gen.make_routing(2000, 8, 16, seed=7, skew=1.2).numpy()
    a = O.build_schedule(te, 16, 0.05)
    b = O.build_schedule(te, 16, 1.0)
    for key in ("cnt", "row0", "row_src", "slot_row"):
        assert (a[key] == b[key]).all()
    ta = sorted(zip(a["tile_expert"], a["tile_row0"], a["tile_rows"]))
    tb = sorted(zip(b["tile_expert"], b["tile_row0"], b["tile_rows"]))
    assert ta == tb
    # c = 1.0 leaves no overflow: the list is expert-ascending
    assert b["num_primary"] == b["num_tiles"]
    nt = b["num_tiles"]
    assert (np.diff(b["tile_expert"][:nt]) >= 0).all()
    # a tiny budget sends the later tiles of hot experts to the overflow part
    assert a["num_primary"] < a["num_tiles"]
    cap = O.capacity_tiles(2000, 0.05, O.max_tiles(2000, 8, 16))
    assert cap == math.ceil(math.ceil(0.05 * 2000) / 128)
    per_e = np.bincount(a["tile_expert"][: a["num_primary"]], minlength=16)
    assert per_e.max() <= cap


def test_schedule_rejects_out_of_range_expert():
    te = np.zeros((4, 2), np.int64)
    te[2, 1] = 9
    assert O.build_schedule(te, 8)["status"] == O.STATUS_INDEX
    te[2, 1] = -1
    assert O.build_schedule(te, 8)["status"] == O.STATUS_INDEX


# ------------------------------------------------------------------ E4M3 / E8M0

def test_e4m3_anchor_values_from_format_spec():
    for code, val in _read_pairs("e4m3_anchors.txt"):
        c = int(code, 16)
        v = O.e4m3_decode(np.array([c], np.uint8))[0]
        if val == "nan":
            assert np.isnan(v)
        else:
            assert v == float(val) and np.signbit(v) == val.startswith("-")
            assert O.e4m3_encode(np.array([float(val)]))[0] == c


def test_e8m0_anchor_values_from_format_spec():
    for code, ex in _read_pairs("e8m0_anchors.txt"):
        # a block whose amax is exactly 448 * 2^ex gets exponent ex
        amax = 448.0 * 2.0 ** int(ex)
        assert O.e8m0_scale_exponent(np.array([amax]))[0] + 127 == int(code)


def test_worked_block_example():
    rows = _read_pairs("mxfp8_block_example.txt")
    vals = [float(v) for v, _ in rows]
    codes = [int(c, 16) for _, c in rows]
    block = np.array(vals + [0.5] * (32 - len(vals)))
    q, s = O.mxfp8_quantize(block[None, :])
    assert s[0, 0] == 120
    assert list(q[0, : len(vals)]) == codes
    assert (q[0, len(vals):] == 0x68).all()


def _table():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    return codes, O.e4m3_decode(codes)


def test_e4m3_roundtrip_all_codes():
    codes, vals = _table()
    assert (O.e4m3_encode(vals) == codes).all()


def _brute_nearest(v, codes, vals):
    """Nearest finite E4M3 code; ties go to the code with an even mantissa;
    saturate beyond 448; zero keeps the sign of v."""
    a = min(abs(v), 448.0)
    pos = vals >= 0
    pc, pv = codes[pos & ~np.signbit(vals)], vals[pos & ~np.signbit(vals)]
    d = np.abs(pv - a)
    best = np.flatnonzero(d == d.min())
    if len(best) > 1:
        best = [b for b in best if (pc[b] & 1) == 0]
    c = int(pc[best[0]])
    return c | (0x80 if np.signbit(v) else 0)


def test_e4m3_encode_matches_brute_force():
    codes, vals = _table()
    rng = np.random.default_rng(0)
    fin = vals[np.isfinite(vals)]
    mids = (np.sort(np.unique(np.abs(fin)))[1:] + np.sort(np.unique(np.abs(fin)))[:-1]) / 2
    samples = np.concatenate([
        rng.normal(size=3000) * 50, rng.uniform(-500, 500, 2000),
        rng.normal(size=1000) * 0.01, mids, -mids, [0.0, -0.0, 1e-30, -1e-30, 447.9, 460.0],
    ])
    got = O.e4m3_encode(samples)
    want = np.array([_brute_nearest(v, codes, vals) for v in samples], np.uint8)
    assert (got == want).all()


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.normal(size=20000) * 30, rng.normal(size=5000) * 0.003])
    v = v[np.abs(v) <= 448]
    t = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn)
    want = t.view(torch.uint8).numpy()
    # compare values (fp32 input for torch; fp64 for the oracle gives the same
    # rounding unless a value sits within fp32 precision of a midpoint)
    v32 = v.astype(np.float32).astype(np.float64)
    assert (O.e4m3_encode(v32) == want).all()


def test_e8m0_matches_brute_force():
    rng = np.random.default_rng(2)
    amax = np.concatenate([np.abs(rng.normal(size=2000)) * 10.0 ** rng.uniform(-40, 38, 2000),
                           [448.0, 448.0 * 2 ** -3, 448.0001, 1e-45, 3e38, 0.0]])
    got = O.e8m0_scale_exponent(amax)
    for a, s in zip(amax, got):
        if a == 0:
            assert s == 0
            continue
        want = next(x for x in range(-127, 128) if a <= 448.0 * 2.0 ** x or x == 127)
        assert s == want, (a, s, want)


def test_mxfp8_quantize_invariants():
    x = gen.make_matrix(64, 256, std=3.0, seed=3).double().numpy()
    x[3, :32] = 0.0
    x[5, 32:64] *= 1e-30
    q, s = O.mxfp8_quantize(x)
    assert q.dtype == np.uint8 and s.shape == (64, 8)
    assert s[3, 0] == 127 and (q[3, :32] == 0).all()
    y = O.mxfp8_dequantize(q, s)
    # every block: |x / 2^s| <= 448 and the decoded values are within half a quantum
    sc = 2.0 ** (s.astype(np.int64) - 127)
    xb = np.abs(x.reshape(64, 8, 32)) / sc[:, :, None]
    assert xb.max() <= 448.0
    rel = np.abs(y - x).reshape(64, 8, 32) / sc[:, :, None]
    assert (rel <= np.maximum(np.abs(xb) * 2 ** -4, 2 ** -10) + 1e-12).all()
    # idempotent in value: re-quantising the dequantised values changes
    # nothing; the codes repeat wherever the block scale is unchanged (a block
    # whose amax rounded down to 224 * 2^s drops to scale 2^(s-1))
    q2, s2 = O.mxfp8_quantize(y)
    assert (O.mxfp8_dequantize(q2, s2) == y).all()
    same = np.repeat(s2 == s, 32, axis=1)
    assert (q2[same] == q[same]).all()


# ------------------------------------------------------------------ forward

def _tiny(T=16, H=32, I=32, E=4, k=2, I_s=0, seed=0):
    return gen.make_layer_inputs(T, H, I, E, k, I_s, seed=seed)


def _args(inp):
    return (inp.x, inp.router_w, inp.top_experts, inp.w_gate, inp.w_up, inp.w_down,
            inp.ws_gate, inp.ws_up, inp.ws_down)


def test_forward_reduces_to_dense_swiglu_mlp():
    """k = 1, every token on expert 0 with weight 1: the layer is one dense
    SwiGLU MLP, computed here with torch.matmul in float64."""
    inp = _tiny(T=24, H=64, I=96, E=3, k=1)
    top = torch.zeros(24, 1, dtype=torch.int64)
    w = torch.ones(24, 1)
    y = O.layer_forward(inp.x, w, top, inp.w_gate, inp.w_up, inp.w_down)
    x = inp.x.double()
    g = torch.matmul(x, inp.w_gate[0].double().t())
    u = torch.matmul(x, inp.w_up[0].double().t())
    ref = torch.matmul(torch.nn.functional.silu(g) * u, inp.w_down[0].double().t())
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_forward_matches_per_token_loop():
    inp = _tiny(T=10, H=16, I=24, E=5, k=3, I_s=8, seed=4)
    y = O.layer_forward(*_args(inp))
    x = inp.x.double().numpy()
    wg, wu, wd = (a.double().numpy() for a in (inp.w_gate, inp.w_up, inp.w_down))
    sg, su, sd = (a.double().numpy() for a in (inp.ws_gate, inp.ws_up, inp.ws_down))
    for t in range(10):
        acc = np.zeros(16)
        for i in range(16):                       # shared expert, scalar loops
            s = 0.0
            for m in range(8):
                gm = sum(sg[m, h] * x[t, h] for h in range(16))
                um = sum(su[m, h] * x[t, h] for h in range(16))
                s += sd[i, m] * (gm / (1 + math.exp(-gm))) * um
            acc[i] += s
        for j in range(3):
            e = int(inp.top_experts[t, j])
            wt = float(inp.router_w[t, j])
            hv = [(lambda gm, um: gm / (1 + math.exp(-gm)) * um)(
                sum(wg[e, m, h] * x[t, h] for h in range(16)),
                sum(wu[e, m, h] * x[t, h] for h in range(16))) for m in range(24)]
            for i in range(16):
                acc[i] += wt * sum(wd[e, i, m] * hv[m] for m in range(24))
        np.testing.assert_allclose(y[t], acc, rtol=1e-10, atol=1e-12)


def test_forward_zero_router_weights_leaves_shared_expert():
    inp = _tiny(I_s=16, seed=5)
    y = O.layer_forward(inp.x, torch.zeros_like(inp.router_w), inp.top_experts,
                        inp.w_gate, inp.w_up, inp.w_down, inp.ws_gate, inp.ws_up, inp.ws_down)
    x = inp.x.double()
    ref = torch.matmul(torch.nn.functional.silu(x @ inp.ws_gate.double().t()) *
                       (x @ inp.ws_up.double().t()), inp.ws_down.double().t())
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_forward_linear_in_router_weights():
    inp = _tiny(seed=6)
    a = O.layer_forward(*_args(inp))
    w2 = inp.router_w * 4.0  # a power of two keeps the fp32 weights exact
    b = O.layer_forward(inp.x, w2, inp.top_experts, inp.w_gate, inp.w_up, inp.w_down)
    np.testing.assert_allclose(b, 4.0 * a, rtol=1e-12, atol=1e-13)


def test_forward_token_permutation_equivariant():
    inp = _tiny(T=20, I_s=8, seed=7)
    perm = torch.randperm(20, generator=torch.Generator().manual_seed(0))
    a = O.layer_forward(*_args(inp))
    b = O.layer_forward(inp.x[perm], inp.router_w[perm], inp.top_experts[perm], inp.w_gate,
                        inp.w_up, inp.w_down, inp.ws_gate, inp.ws_up, inp.ws_down)
    np.testing.assert_allclose(b, a[perm.numpy()], rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ backward

def _loss(inp_arrays, dy):
    y = O.layer_forward(*inp_arrays)
    return float(np.sum(y * dy))


@pytest.mark.parametrize("shared", [False, True])
def test_backward_matches_finite_differences(shared):
    inp = _tiny(T=6, H=32, I=32, E=4, k=2, I_s=16 if shared else 0, seed=8)
    dy = inp.dy.double().numpy()
    g = O.layer_backward(*_args(inp)[:6], inp.dy, *_args(inp)[6:])
    arrays = [a.double().numpy() if a is not None and a.dtype != torch.int64 else
              (a.numpy() if a is not None else None) for a in _args(inp)]
    rng = np.random.default_rng(0)
    names = {0: "dx", 1: "d_router_w", 3: "d_w_gate", 4: "d_w_up", 5: "d_w_down",
             6: "d_ws_gate", 7: "d_ws_up", 8: "d_ws_down"}
    eps = 1e-5
    for idx, key in names.items():
        if arrays[idx] is None:
            continue
        for _ in range(6):
            pos = tuple(rng.integers(0, s) for s in arrays[idx].shape)
            plus = [a.copy() if isinstance(a, np.ndarray) else a for a in arrays]
            minus = [a.copy() if isinstance(a, np.ndarray) else a for a in arrays]
            plus[idx][pos] += eps
            minus[idx][pos] -= eps
            fd = (_loss(plus, dy) - _loss(minus, dy)) / (2 * eps)
            an = g[key][pos]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (key, pos, fd, an)


def test_router_grad_is_dot_of_dy_with_expert_output():
    """d_w[t, j] = <dy[t], F_e(x[t])> = <W_down^T dy[t], h>: both sides of the
    identity the GPU's down-projection backward uses."""
    inp = _tiny(T=8, seed=9)
    g = O.layer_backward(*_args(inp)[:6], inp.dy)
    x = inp.x.double().numpy()
    dy = inp.dy.double().numpy()
    for t in range(8):
        for j in range(2):
            e = int(inp.top_experts[t, j])
            wg, wu, wd = (a[e].double().numpy() for a in (inp.w_gate, inp.w_up, inp.w_down))
            h = O.silu(wg @ x[t]) * (wu @ x[t])
            lhs = dy[t] @ (wd @ h)
            rhs = (wd.T @ dy[t]) @ h
            assert abs(lhs - g["d_router_w"][t, j]) < 1e-12
            assert abs(rhs - lhs) < 1e-12


# ------------------------------------------------------------------ MXFP8 layer

def _brute_q(v):
    """Brute-force MXFP8 round trip of one vector, block by block, using the
    code table and the brute-force nearest-code search."""
    codes, vals = _table()
    out = np.empty_like(v)
    for b in range(0, len(v), 32):
        blk = v[b:b + 32]
        amax = np.abs(blk).max()
        s = 0 if amax == 0 else next(x for x in range(-127, 128) if amax <= 448.0 * 2.0 ** x)
        for i, a in enumerate(blk):
            c = _brute_nearest(a * 2.0 ** -s, codes, vals)
            out[b + i] = O.e4m3_decode(np.array([c], np.uint8))[0] * 2.0 ** s
    return out


def test_mxfp8_forward_matches_per_token_brute_force():
    inp = _tiny(T=4, H=64, I=64, E=3, k=2, I_s=32, seed=10)
    y = O.layer_forward_mxfp8(*_args(inp))
    x = inp.x.double().numpy()

    def qrows(m):
        return np.stack([_brute_q(r) for r in m])

    def expert(v, wg, wu, wd):
        g = qrows(wg) @ v
        u = qrows(wu) @ v
        h = _brute_q(O.silu(g) * u)
        return qrows(wd) @ h

    for t in range(4):
        xq = _brute_q(x[t])
        acc = expert(xq, inp.ws_gate.double().numpy(), inp.ws_up.double().numpy(),
                     inp.ws_down.double().numpy())
        for j in range(2):
            e = int(inp.top_experts[t, j])
            acc = acc + float(inp.router_w[t, j]) * expert(
                xq, inp.w_gate[e].double().numpy(), inp.w_up[e].double().numpy(),
                inp.w_down[e].double().numpy())
        np.testing.assert_allclose(y[t], acc, rtol=1e-10, atol=1e-12)


def test_mxfp8_backward_equals_bf16_backward_on_grid_inputs():
    """When x and the gate/up weights already lie on the MXFP8 grid, the
    quantised forward's gate/up pre-activations equal the unquantised ones,
    so the straight-through backward must equal the exact BF16 backward."""
    inp = _tiny(T=8, H=64, I=32, E=3, k=2, I_s=32, seed=11)
    for name in ("x", "w_gate", "w_up", "ws_gate", "ws_up"):
        t = getattr(inp, name)
        flat = t.double().reshape(-1, t.shape[-1]).numpy()
        setattr(inp, name, torch.from_numpy(O.mxfp8_roundtrip(flat)).reshape(t.shape))
    a = O.layer_backward_mxfp8(*_args(inp)[:6], inp.dy, *_args(inp)[6:])
    b = O.layer_backward(*_args(inp)[:6], inp.dy, *_args(inp)[6:])
    for key in b:
        np.testing.assert_allclose(a[key], b[key], rtol=1e-12, atol=1e-14)


def _brute_mxfp8_backward(inp):
    """The straight-through backward of the MXFP8 forward, token by token in
    plain Python floats: the gate/up pre-activations from the brute-force
    quantised x and gate/up weight rows; everything after them (the SwiGLU
    derivative, dx, the weight gradients, <dy, F(x)>) with the bf16 weights
    and the unquantised x."""
    x = inp.x.double().tolist()
    dy = inp.dy.double().tolist()
    rw = inp.router_w.double().tolist()
    te = inp.top_experts.tolist()
    T, H, k = len(x), len(x[0]), len(te[0])
    E, I = inp.w_gate.shape[0], inp.w_gate.shape[1]
    out = {"dx": [[0.0] * H for _ in range(T)], "d_router_w": [[0.0] * k for _ in range(T)],
           "d_w_gate": np.zeros((E, I, H)), "d_w_up": np.zeros((E, I, H)), "d_w_down": np.zeros((E, H, I))}
    if inp.ws_gate is not None:
        Is = inp.ws_gate.shape[0]
        out.update(d_ws_gate=np.zeros((Is, H)), d_ws_up=np.zeros((Is, H)), d_ws_down=np.zeros((H, Is)))
    qcache = {}

    def qrows(key, m):
        if key not in qcache:
            qcache[key] = [list(_brute_q(np.asarray(r))) for r in m]
        return qcache[key]

    def expert(t, key, wg, wu, wd, scale, dWg, dWu, dWd):
        xq = list(_brute_q(np.asarray(x[t])))
        qg, qu = qrows((key, "g"), wg), qrows((key, "u"), wu)
        n_i = len(wg)
        g = [sum(a * b for a, b in zip(qg[i], xq)) for i in range(n_i)]
        u = [sum(a * b for a, b in zip(qu[i], xq)) for i in range(n_i)]
        sg = [1.0 / (1.0 + math.exp(-v)) for v in g]
        h = [g[i] * sg[i] * u[i] for i in range(n_i)]
        dot = sum(dy[t][r] * sum(wd[r][i] * h[i] for i in range(n_i)) for r in range(H))
        for i in range(n_i):
            z = sum(wd[r][i] * dy[t][r] for r in range(H))
            dh = scale * z
            dg = dh * u[i] * sg[i] * (1.0 + g[i] * (1.0 - sg[i]))
            du = dh * g[i] * sg[i]
            for c in range(H):
                out["dx"][t][c] += dg * wg[i][c] + du * wu[i][c]
                dWg[i, c] += dg * x[t][c]
                dWu[i, c] += du * x[t][c]
                dWd[c, i] += scale * dy[t][c] * h[i]
        return dot

    for t in range(T):
        if inp.ws_gate is not None:
            expert(t, "s", inp.ws_gate.double().tolist(), inp.ws_up.double().tolist(),
                   inp.ws_down.double().tolist(), 1.0, out["d_ws_gate"], out["d_ws_up"], out["d_ws_down"])
        for j in range(k):
            e = te[t][j]
            out["d_router_w"][t][j] = expert(
                t, e, inp.w_gate[e].double().tolist(), inp.w_up[e].double().tolist(),
                inp.w_down[e].double().tolist(), rw[t][j], out["d_w_gate"][e], out["d_w_up"][e], out["d_w_down"][e])
    return {key: np.asarray(v) for key, v in out.items()}


def test_mxfp8_backward_matches_per_token_brute_force():
    """The MXFP8-forward layer's BF16 backward (straight-through, taken at the
    quantised forward's pre-activations) against its per-token restatement."""
    inp = _tiny(T=4, H=64, I=32, E=3, k=2, I_s=32, seed=14)
    got = O.layer_backward_mxfp8(*_args(inp)[:6], inp.dy, *_args(inp)[6:])
    ref = _brute_mxfp8_backward(inp)
    assert set(got) == set(ref)
    for key in ref:
        np.testing.assert_allclose(got[key], ref[key], rtol=1e-9, atol=1e-13, err_msg=key)


def test_mxfp8_backward_pin_rejects_other_evaluation_points():
    """Planted mistakes, in copies of the oracle's MXFP8 backward: the
    derivative taken at the unquantised pre-activations, or with only x or
    only the weights quantised.  Each must miss the per-token restatement."""
    inp = _tiny(T=4, H=64, I=32, E=3, k=2, I_s=32, seed=14)
    ref = _brute_mxfp8_backward(inp)
    a = _args(inp)
    wg, wu = inp.w_gate.double().numpy(), inp.w_up.double().numpy()
    sg, su = inp.ws_gate.double().numpy(), inp.ws_up.double().numpy()

    def mutant(qx, qw):
        def gu(e, v):
            vv = O.mxfp8_roundtrip(v) if qx else v
            mg, mu = (sg, su) if e is None else (wg[e], wu[e])
            if qw:
                mg, mu = O.mxfp8_roundtrip(mg), O.mxfp8_roundtrip(mu)
            return vv @ mg.T, vv @ mu.T
        return O.layer_backward(*a[:6], inp.dy, *a[6:], gu_override=gu)

    for qx, qw in ((False, False), (True, False), (False, True)):
        bad = mutant(qx, qw)
        assert not np.allclose(bad["dx"], ref["dx"], rtol=1e-6, atol=1e-9), (qx, qw)
    # the same construction with both quantised passes (the copies are faithful)
    good = mutant(True, True)
    for key in ref:
        np.testing.assert_allclose(good[key], ref[key], rtol=1e-9, atol=1e-13, err_msg=key)


def test_capacity_budget_is_rounded_up_in_double_precision():
    """c*T rounded up on the float64 value of the multiplier: 0.05 * 2560 is
    128 rows (one tile), although float32(0.05) * 2560 is just above 128."""
    assert O.capacity_tiles(2560, 0.05, 1000) == 1
    assert O.capacity_tiles(1280, 0.3, 1000) == 3
    assert O.capacity_tiles(2560, 0.0501, 1000) == 2
    assert O.capacity_tiles(100, 50.0, 7) == 7          # never above the tile bound


def test_mxfp8_forward_close_to_unquantised():
    inp = _tiny(T=32, H=64, I=64, E=4, k=2, seed=12)
    a = O.layer_forward_mxfp8(*_args(inp))
    b = O.layer_forward(*_args(inp))
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert 1e-3 < rel < 0.1


# ------------------------------------------------------------------ swiglu_limit

def _gate_up_values(inp):
    """Every gate and |up| pre-activation value the layer forms (test helper
    for choosing a clamp limit away from all of them)."""
    x = inp.x.double().numpy()
    vals = []
    te = inp.top_experts.numpy()
    for t in range(x.shape[0]):
        for e in te[t]:
            vals += list(inp.w_gate[e].double().numpy() @ x[t])
            vals += list(np.abs(inp.w_up[e].double().numpy() @ x[t]))
    if inp.ws_gate is not None:
        vals += list((x @ inp.ws_gate.double().numpy().T).ravel())
        vals += list(np.abs(x @ inp.ws_up.double().numpy().T).ravel())
    return np.sort(np.asarray(vals))


def _limit_between(vals, lo_q=0.6, hi_q=0.9):
    """A limit in the widest gap between consecutive values of the given
    quantile range (so a central difference never crosses a clamp kink),
    where moreover every value and its bf16 rounding fall on the same side of
    the limit; returns the limit and the distance to the nearest value."""
    a = vals[int(lo_q * len(vals)):int(hi_q * len(vals))]
    for i in np.argsort(-np.diff(a)):
        L = float(np.float32(0.5 * (a[i] + a[i + 1])))
        if np.array_equal(vals <= L, O.round_bf16(vals) <= L):
            return L, 0.5 * (a[i + 1] - a[i])
    raise AssertionError("no limit with consistent bf16 decisions")


def test_round_bf16_matches_torch_cast():
    """The oracle's bf16 rounding (float32 bits, ties to even) against
    torch's float32 -> bfloat16 conversion, over wide magnitudes and exact
    ties."""
    rng = np.random.default_rng(5)
    x = rng.normal(size=50000) * np.exp(rng.normal(size=50000) * 4)
    ties = (np.arange(1, 2001, dtype=np.uint32) << 16 | 0x8000).view(np.float32).astype(np.float64)
    for v in (x, ties, -ties):
        ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).double().numpy()
        assert np.array_equal(O.round_bf16(v), ref)


def test_swiglu_limit_off_and_huge_equal_the_plain_layer():
    inp = _tiny(T=12, H=32, I=32, E=4, k=2, I_s=16, seed=21)
    a = _args(inp)
    y0 = O.layer_forward(*a)
    assert np.array_equal(O.layer_forward(*a, swiglu_limit=0.0), y0)
    assert np.array_equal(O.layer_forward(*a, swiglu_limit=1e30), y0)
    g0 = O.layer_backward(*a[:6], inp.dy, *a[6:])
    g1 = O.layer_backward(*a[:6], inp.dy, *a[6:], swiglu_limit=1e30)
    for key in g0:
        assert np.array_equal(g0[key], g1[key]), key


def test_swiglu_limit_matches_per_token_scalar_loop():
    """With a limit that clamps a good share of the pre-activations, the layer
    equals a per-token loop in plain Python floats, the clamp written as
    comparisons."""
    inp = _tiny(T=6, H=16, I=12, E=3, k=2, I_s=8, seed=22)
    vals = _gate_up_values(inp)
    L = float(np.quantile(vals, 0.7))
    y = O.layer_forward(*_args(inp), swiglu_limit=L)
    x = inp.x.double().tolist()
    rw = inp.router_w.double().tolist()
    te = inp.top_experts.tolist()
    clamped = 0

    def expert(v, wg, wu, wd, scale, acc):
        nonlocal clamped
        for i in range(len(wg)):
            g = sum(a * b for a, b in zip(v, wg[i]))
            u = sum(a * b for a, b in zip(v, wu[i]))
            if g > L:
                g, clamped = L, clamped + 1
            if u > L:
                u, clamped = L, clamped + 1
            elif u < -L:
                u, clamped = -L, clamped + 1
            h = g / (1.0 + math.exp(-g)) * u
            for r in range(len(acc)):
                acc[r] += scale * wd[r][i] * h

    sg, su, sd = (a.double().tolist() for a in (inp.ws_gate, inp.ws_up, inp.ws_down))
    for t in range(6):
        acc = [0.0] * 16
        expert(x[t], sg, su, sd, 1.0, acc)
        for j in range(2):
            e = te[t][j]
            expert(x[t], inp.w_gate[e].double().tolist(), inp.w_up[e].double().tolist(),
                   inp.w_down[e].double().tolist(), rw[t][j], acc)
        np.testing.assert_allclose(y[t], acc, rtol=1e-12, atol=1e-14)
    assert clamped > 20


@pytest.mark.parametrize("shared", [False, True])
def test_swiglu_limit_backward_matches_finite_differences(shared):
    """Central differences of the clamped layer, with the limit placed between
    pre-activation values (so no perturbation crosses a clamp kink): the
    analytic gradients, masked where the clamp holds, must match."""
    inp = _tiny(T=6, H=32, I=32, E=4, k=2, I_s=16 if shared else 0, seed=23)
    vals = _gate_up_values(inp)
    L, margin = _limit_between(vals)
    assert margin > 1e-4 and np.mean(vals > L) > 0.05     # the clamp is active somewhere
    dy = inp.dy.double().numpy()
    a = _args(inp)
    g = O.layer_backward(*a[:6], inp.dy, *a[6:], swiglu_limit=L)
    arrays = [v.double().numpy() if v is not None and v.dtype != torch.int64 else
              (v.numpy() if v is not None else None) for v in a]
    rng = np.random.default_rng(1)
    names = {0: "dx", 1: "d_router_w", 3: "d_w_gate", 4: "d_w_up", 5: "d_w_down",
             6: "d_ws_gate", 7: "d_ws_up", 8: "d_ws_down"}
    eps = 1e-6

    def loss(arrs):
        return float(np.sum(O.layer_forward(*arrs, swiglu_limit=L) * dy))

    for idx, key in names.items():
        if arrays[idx] is None:
            continue
        for _ in range(8):
            pos = tuple(rng.integers(0, s) for s in arrays[idx].shape)
            plus = [v.copy() if isinstance(v, np.ndarray) else v for v in arrays]
            minus = [v.copy() if isinstance(v, np.ndarray) else v for v in arrays]
            plus[idx][pos] += eps
            minus[idx][pos] -= eps
            fd = (loss(plus) - loss(minus)) / (2 * eps)
            an = g[key][pos]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (key, pos, fd, an)
    # the mask matters: the unclamped gradients differ
    g_plain = O.layer_backward(*a[:6], inp.dy, *a[6:])
    assert not np.allclose(g_plain["dx"], g["dx"])


# ------------------------------------------------------------------ MXFP8 backward

def _bf16_torch(a):
    """bf16 rounding through torch casts (float64 -> float32 -> bfloat16)."""
    return torch.from_numpy(np.asarray(a, np.float64)).float().bfloat16().double().numpy()


def test_mxfp8_full_backward_matches_brute_force():
    """Every backward GEMM operand quantised by the brute-force codec, vector
    by vector along the axis the reading names (rows of dy and dG|dU; columns
    of W_down along H and of W_gate, W_up along I; columns of the weight
    gradients' operands over 32-row groups of each expert's rows, taken in
    ascending f), then contracted by explicit scalar sums."""
    T, H, I, E, k, Is = 24, 64, 32, 2, 2, 32
    inp = _tiny(T=T, H=H, I=I, E=E, k=k, I_s=Is, seed=13)
    got = O.layer_backward_mxfp8_full(*_args(inp)[:6], inp.dy, *_args(inp)[6:])
    x, dy = inp.x.double().numpy(), inp.dy.double().numpy()
    te, rw = inp.top_experts.numpy(), inp.router_w.double().numpy()

    def q_vec_rows(m):           # quantise each row of m (blocks along the row)
        return np.stack([_brute_q(r) for r in m])

    def q_vec_cols(m):           # quantise each column of m (blocks down the column)
        n = m.shape[0]
        pad = (-n) % 32
        out = np.empty_like(m)
        for c in range(m.shape[1]):
            col = np.concatenate([m[:, c], np.zeros(pad)])
            out[:, c] = _brute_q(col)[:n]
        return out

    def dot(a, b):
        return sum(a[i] * b[i] for i in range(len(a)))

    def expert_bwd(rows, wts, Wg, Wu, Wd):
        n, Iw = len(rows), Wg.shape[0]
        v, d = x[rows], dy[rows]
        vq, dq = q_vec_rows(v), q_vec_rows(d)
        Wgq, Wuq = q_vec_rows(Wg), q_vec_rows(Wu)          # forward: along H
        Wdc = q_vec_cols(Wd)                               # dgrad through down: along H
        Wgc, Wuc = q_vec_cols(Wg), q_vec_cols(Wu)          # dgrad through gate/up: along I
        dsc = np.zeros(n)
        dg, du, hw = np.zeros((n, Iw)), np.zeros((n, Iw)), np.zeros((n, Iw))
        for r in range(n):
            for i in range(Iw):
                g = _bf16_torch(dot(vq[r], Wgq[i]))
                u = _bf16_torch(dot(vq[r], Wuq[i]))
                s = 1.0 / (1.0 + math.exp(-g))
                z = dot(dq[r], Wdc[:, i])
                h = g * s * u
                dsc[r] += z * h
                dg[r, i] = wts[r] * z * u * s * (1.0 + g * (1.0 - s))
                du[r, i] = wts[r] * z * g * s
                hw[r, i] = wts[r] * h
        dg, du, hw = _bf16_torch(dg), _bf16_torch(du), _bf16_torch(hw)
        dgq, duq = q_vec_rows(dg), q_vec_rows(du)
        dv = np.array([[dot(dgq[r], Wgc[:, c]) + dot(duq[r], Wuc[:, c]) for c in range(H)] for r in range(n)])
        dc, hc, gc_, uc_, vc = (q_vec_cols(a) for a in (d, hw, dg, du, v))
        dWd = np.array([[dot(dc[:, a], hc[:, b]) for b in range(Iw)] for a in range(H)])
        dWg = np.array([[dot(gc_[:, a], vc[:, b]) for b in range(H)] for a in range(Iw)])
        dWu = np.array([[dot(uc_[:, a], vc[:, b]) for b in range(H)] for a in range(Iw)])
        return dsc, dv, dWg, dWu, dWd

    dx = np.zeros((T, H))
    dsc, dv, dWg, dWu, dWd = expert_bwd(list(range(T)), np.ones(T), inp.ws_gate.double().numpy(),
                                        inp.ws_up.double().numpy(), inp.ws_down.double().numpy())
    dx += dv
    for key, want in (("d_ws_gate", dWg), ("d_ws_up", dWu), ("d_ws_down", dWd)):
        np.testing.assert_allclose(got[key], want, rtol=1e-9, atol=1e-12)
    for e in range(E):
        fl = sorted(t * k + j for t in range(T) for j in range(k) if te[t, j] == e)
        rows = [f // k for f in fl]
        wts = np.array([rw[f // k, f % k] for f in fl])
        dsc, dv, dWg, dWu, dWd = expert_bwd(rows, wts, inp.w_gate[e].double().numpy(),
                                            inp.w_up[e].double().numpy(), inp.w_down[e].double().numpy())
        for n, f in enumerate(fl):
            dx[f // k] += dv[n]
            np.testing.assert_allclose(got["d_router_w"][f // k, f % k], dsc[n], rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(got["d_w_gate"][e], dWg, rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(got["d_w_up"][e], dWu, rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(got["d_w_down"][e], dWd, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(got["dx"], dx, rtol=1e-9, atol=1e-12)


def test_mxfp8_full_backward_scales_with_dy_by_powers_of_two():
    """Scaling dy by 2^5 scales every gradient by exactly 2^5: every
    quantiser commutes with power-of-two scaling (the block scale absorbs
    it) and the bf16 roundings do too."""
    inp = _tiny(T=20, H=64, I=64, E=3, k=2, I_s=32, seed=14)
    a = O.layer_backward_mxfp8_full(*_args(inp)[:6], inp.dy, *_args(inp)[6:])
    b = O.layer_backward_mxfp8_full(*_args(inp)[:6], inp.dy.double() * 32.0, *_args(inp)[6:])
    for key in a:
        np.testing.assert_array_equal(b[key], 32.0 * a[key])


def test_mxfp8_full_backward_close_to_straight_through_bf16_backward():
    """The quantised backward stays within the MXFP8 error of the bf16
    backward of the same quantised forward, output by output."""
    inp = _tiny(T=64, H=128, I=64, E=4, k=2, I_s=64, seed=15)
    a = O.layer_backward_mxfp8_full(*_args(inp)[:6], inp.dy, *_args(inp)[6:])
    b = O.layer_backward_mxfp8(*_args(inp)[:6], inp.dy, *_args(inp)[6:])
    for key in b:
        rel = np.linalg.norm(a[key] - b[key]) / np.linalg.norm(b[key])
        assert 3e-3 < rel < 0.12, (key, rel)
