"""GPU tests of aq_chain_run: every matmul of a chain against the oracle, and
the ordering guarantee (a matmul that reads an earlier matmul's output sees
it completely written)."""
import numpy as np
import pytest

import affine_bit_quantized_gb300 as aq
import oracle
from affine_bit_quantized_gb300 import _build, synth

from ._helpers import assert_parity, from_dev_bf16, to_dev_bf16, to_dev_u32, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    _build.build_library()
    return torch.device("cuda:0")


def _mat(dev, M, N, K, seed, bits=4):
    import torch
    w = synth.make_weights(N, K, seed, bits=bits)
    x = synth.make_x(M, K, seed)
    xt, wt, st, bt = upload(x, w, dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    return x, w, (xt, wt, st, bt, y)


@pytest.mark.parametrize("shapes", [
    [(1, 64, 512)],
    [(1, 4096, 4096), (1, 1024, 4096), (1, 1024, 4096), (1, 4096, 4096), (1, 14336, 4096), (1, 4096, 14336)],
    [(1, 17, 1024), (1, 300, 2560), (1, 1, 512), (1, 1000, 8192), (1, 33, 16384)],
    [(2, 100, 1024), (8, 77, 2048), (3, 15, 512), (1, 260, 1536)],      # M > 1 in the chain: general path
])
def test_chain_parity(dev, shapes):
    import torch
    mats = [_mat(dev, M, N, K, 40 + i) for i, (M, N, K) in enumerate(shapes)]
    chain = aq.Chain([m[2] for m in mats])
    chain.run()
    torch.cuda.synchronize()
    assert aq.aq_read_device_status(None) == aq.AQ_OK
    for (x, w, t), (M, N, K) in zip(mats, shapes):
        _, ref = oracle.matmul(x, w.w_packed, w.scales, w.biases, M, N, K)
        assert_parity(from_dev_bf16(t[4]), ref, what=f"chain M={M} N={N} K={K}")


def test_chain_same_bits_as_single_calls_and_repeatable(dev):
    import torch
    shapes = [(1, 4096, 4096), (1, 1024, 4096), (1, 14336, 4096)]
    mats = [_mat(dev, M, N, K, 60 + i) for i, (M, N, K) in enumerate(shapes)]
    chain = aq.Chain([m[2] for m in mats])
    chain.run()
    torch.cuda.synchronize()
    first = [m[2][4].clone() for m in mats]
    chain.run()
    chain.run()
    torch.cuda.synchronize()
    for m, f in zip(mats, first):
        xt, wt, st, bt, y = m[2]
        assert torch.equal(y, f)
        assert torch.equal(y, aq.matmul(xt, wt, st, bt))


def test_chain_dependency_reads_earlier_output(dev):
    """x of matmul j+1 IS the output buffer of matmul j.  The chain must give
    exactly what a sequence of separate calls gives (each call sees the
    previous output completely written)."""
    import torch
    Ks = [512, 1024, 2048, 1024, 4096]   # N of matmul j = K of matmul j+1
    Ns = Ks[1:] + [3000]
    ws = [synth.make_weights(N, K, 70 + i) for i, (N, K) in enumerate(zip(Ns, Ks))]
    x0 = to_dev_bf16(synth.make_x(1, Ks[0], 70), dev)
    wdev = [upload(np.zeros((1, w.K), np.uint16), w, dev)[1:] for w in ws]
    ys = [torch.empty((1, N), dtype=torch.bfloat16, device=dev) for N in Ns]
    items = []
    for i in range(len(ws)):
        xin = x0 if i == 0 else ys[i - 1]
        items.append((xin, *wdev[i], ys[i]))
    chain = aq.Chain(items)
    for _ in range(3):
        for y in ys:
            y.fill_(float("nan"))
        chain.run()
        torch.cuda.synchronize()
        # reference: separate calls, in order
        cur = x0
        for i in range(len(ws)):
            ref = aq.matmul(cur, *wdev[i])
            torch.cuda.synchronize()
            assert torch.equal(ys[i], ref), f"matmul {i}"
            cur = ref


def test_chain_independent_matmuls_share_x(dev):
    """q, k, v read one x and do not depend on each other (k and v flagged
    independent); gate and up likewise; o and down depend on earlier outputs.
    Every output equals the separate-call result bit for bit, and matches the
    oracle."""
    import torch
    K = 1024
    x_attn = synth.make_x(1, K, 81)
    x_mlp = synth.make_x(1, K, 82)
    xa, xm = to_dev_bf16(x_attn, dev), to_dev_bf16(x_mlp, dev)
    # o reads q's output, down reads o's output
    items, indep, refs = [], [], []
    plan = [("q", 512, K, "xa"), ("k", 128, K, "xa"), ("v", 128, K, "xa"), ("o", 1024, 512, "q"),
            ("gate", 700, K, "xm"), ("up", 700, K, "xm"), ("down", 1000, 1024, "o")]
    outs = {}
    for i, (name, N, Kin, src) in enumerate(plan):
        w = synth.make_weights(N, Kin, 90 + i)
        wt = upload(np.zeros((1, Kin), np.uint16), w, dev)[1:]
        y = torch.empty((1, N), dtype=torch.bfloat16, device=dev)
        xin = {"xa": xa, "xm": xm}.get(src, outs.get(src))
        items.append((xin, *wt, y))
        indep.append(name in ("k", "v", "up"))
        outs[name] = y
        refs.append((w, src))
    chain = aq.Chain(items, independent=indep)
    for _ in range(2):
        for it in items:
            it[4].fill_(float("nan"))
        chain.run()
        torch.cuda.synchronize()
        assert aq.aq_read_device_status(None) == aq.AQ_OK
        got = {name: items[i][4].clone() for i, (name, *_r) in enumerate(plan)}
        # separate calls in order give the same bits
        for i, (name, *_r) in enumerate(plan):
            xin, wt, st, bt, y = items[i]
            assert torch.equal(got[name], aq.matmul(xin, wt, st, bt)), name
    # the ones whose input is a host-generated x also match the oracle
    for i, (name, N, Kin, src) in enumerate(plan):
        if src in ("xa", "xm"):
            w = refs[i][0]
            xh = x_attn if src == "xa" else x_mlp
            _, ref = oracle.matmul(xh, w.w_packed, w.scales, w.biases, 1, N, Kin)
            assert_parity(from_dev_bf16(got[name]), ref, what=name)


@pytest.mark.parametrize("shapes", [
    [(1, 4096, 4096), (1, 1024, 4096), (1, 14336, 4096), (1, 4096, 14336)],
    [(1, 17, 1024), (2, 300, 2048), (1, 33, 16384), (4, 50, 1536)],
])
def test_chain_eight_bit(dev, shapes):
    """A chain of 8-bit matmuls: every output against the oracle, and the same
    bits as single calls."""
    import torch
    mats = [_mat(dev, M, N, K, 500 + i, bits=8) for i, (M, N, K) in enumerate(shapes)]
    chain = aq.Chain([m[2] for m in mats], bits=8)
    chain.run()
    torch.cuda.synchronize()
    assert aq.aq_read_device_status(None) == aq.AQ_OK
    for (x, w, t), (M, N, K) in zip(mats, shapes):
        _, ref = oracle.matmul(x, w.w_packed, w.scales, w.biases, M, N, K, bits=8)
        assert_parity(from_dev_bf16(t[4]), ref, what=f"chain 8-bit M={M} N={N} K={K}")
        xt, wt, st, bt, y = t
        assert torch.equal(y, aq.matmul(xt, wt, st, bt, bits=8))


def test_chain_longer_than_the_shared_memory_record_cache(dev):
    """300 matmuls (the kernel keeps the first 256 records' scalars in shared
    memory and reads the rest from global memory): pairs of a dependent matmul
    that reads the previous pair's output and an independent one on the same
    input.  Every output is compared with the oracle on the inputs it actually
    read, and with separate calls bit for bit."""
    import torch
    K = 512
    pairs = 150
    x0 = to_dev_bf16(synth.make_x(1, K, 700), dev)
    items, indep, ws = [], [], []
    prev = x0
    for p in range(pairs):
        for half, N in enumerate((K, 77 + p % 5)):
            w = synth.make_weights(N, K, 1000 + 2 * p + half)
            wt = upload(np.zeros((1, K), np.uint16), w, dev)[1:]
            y = torch.empty((1, N), dtype=torch.bfloat16, device=dev)
            items.append((prev, *wt, y))
            indep.append(half == 1)
            ws.append(w)
        prev = items[-2][4]            # the next pair reads this pair's dependent output
    assert len(items) == 300
    chain = aq.Chain(items, independent=indep)
    for it in items:
        it[4].fill_(float("nan"))
    chain.run()
    torch.cuda.synchronize()
    assert aq.aq_read_device_status(None) == aq.AQ_OK
    for i, ((xin, wt, st, bt, y), w) in enumerate(zip(items, ws)):
        xh = from_dev_bf16(xin).reshape(1, K)
        _, ref = oracle.matmul(xh, w.w_packed, w.scales, w.biases, 1, w.N, K)
        assert_parity(from_dev_bf16(y), ref, what=f"matmul {i}")
        assert torch.equal(y, aq.matmul(xin, wt, st, bt)), f"matmul {i}"


def test_chain_bounded_wait_timeout_reports_status(dev):
    """A matmul flagged with the chain's test hook loses its first copy in the
    first CTA: that CTA's wait expires and it stops, the other CTAs' waits for
    its completion count expire too, the host reads AQ_ERR_TIMEOUT, and a
    normal run of the same chain right after matches the oracle."""
    import torch
    shapes = [(1, 4096, 4096), (1, 1024, 4096), (1, 14336, 4096), (1, 4096, 14336)]
    mats = [_mat(dev, M, N, K, 80 + i) for i, (M, N, K) in enumerate(shapes)]
    stream = torch.cuda.current_stream().cuda_stream

    def descs(hook):
        return (aq.MatmulDesc * len(mats))(*[
            aq.MatmulDesc(t[0].data_ptr(), t[1].data_ptr(), t[2].data_ptr(), t[3].data_ptr(), t[4].data_ptr(), M, N,
                          K, aq.AQ_CHAIN_DEBUG_SKIP_COPY if (hook and i == 1) else 0)
            for i, ((x, w, t), (M, N, K)) in enumerate(zip(mats, shapes))])

    nbytes = aq.aq_chain_workspace_bytes(len(mats))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    for hook in (True, False):
        plan = aq.ChainPlan()
        assert aq.aq_chain_prepare(descs(hook), len(mats), 64, 4, ws.data_ptr(), nbytes, plan) == aq.AQ_OK
        assert aq.aq_chain_run(plan, stream) == aq.AQ_OK
        torch.cuda.synchronize()
        assert aq.aq_read_device_status(stream) == (aq.AQ_ERR_TIMEOUT if hook else aq.AQ_OK)
    for (x, w, t), (M, N, K) in zip(mats, shapes):
        _, ref = oracle.matmul(x, w.w_packed, w.scales, w.biases, M, N, K)
        assert_parity(from_dev_bf16(t[4]), ref, what=f"chain after timeout M={M} N={N} K={K}")


# ---------------------------------------------------------------- NVFP4 chains (group size 16)

def _nv_upload(w, dev):
    import torch
    wt = to_dev_u32(w.w_packed, dev)
    st = torch.from_numpy(np.ascontiguousarray(w.scales)).to(dev)
    gs = torch.tensor([w.global_scale], dtype=torch.float32, device=dev)
    return wt, st, gs


@pytest.mark.parametrize("shapes", [
    [(1, 64, 256)],
    [(1, 4096, 4096), (1, 1024, 4096), (1, 14336, 4096), (1, 4096, 14336)],
    [(1, 17, 1280), (2, 300, 2048), (1, 33, 16384), (4, 50, 2304), (8, 77, 2048), (3, 15, 768)],
])
def test_chain_nvfp4_parity(dev, shapes):
    """A chain of NVFP4 matmuls (E2M1 codes, E4M3 block scales, the tensor
    scale read from device memory): every output against the NVFP4 oracle, and
    the same bits as single aq_matmul_nvfp4_bf16 calls."""
    import torch
    mats = []
    for i, (M, N, K) in enumerate(shapes):
        w = synth.make_nvfp4_weights(N, K, 1500 + i)
        x = synth.make_x(M, K, 1500 + i)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        mats.append((x, w, (to_dev_bf16(x, dev), *_nv_upload(w, dev), y)))
    chain = aq.Chain([m[2] for m in mats], group_size=16, bits=4)
    for m in mats:
        m[2][4].fill_(float("nan"))
    chain.run()
    torch.cuda.synchronize()
    assert aq.aq_read_device_status(None) == aq.AQ_OK
    for (x, w, t), (M, N, K) in zip(mats, shapes):
        _, ref = oracle.nvfp4_matmul(x, w.w_packed, w.scales, w.global_scale, M, N, K)
        assert_parity(from_dev_bf16(t[4]), ref, what=f"nvfp4 chain M={M} N={N} K={K}")
        xt, wt, st, gs, y = t
        assert torch.equal(y, aq.matmul_nvfp4(xt, wt, st, w.global_scale)), f"M={M} N={N} K={K}"


def test_chain_nvfp4_dependencies_and_shared_x(dev):
    """NVFP4 chain with a dependent matmul reading the previous output and
    independent ones sharing an x (k, v after q; up after gate), two rows of x.
    Each output matches the oracle on the input it actually read, separate
    calls bit for bit, and the tensor scale is taken from device memory at run
    time (changing it changes the next run's outputs)."""
    import torch
    M, K = 2, 2048
    plan = [("q", 2048, K, "x"), ("k", 512, K, "x"), ("v", 512, K, "x"), ("o", 2048, 2048, "q"),
            ("gate", 1536, 2048, "o"), ("up", 1536, 2048, "o"), ("down", 1000, 1536, "gate")]
    x0 = to_dev_bf16(synth.make_x(M, K, 1600), dev)
    items, indep, ws, outs = [], [], [], {"x": x0}
    for i, (name, N, Kin, src) in enumerate(plan):
        w = synth.make_nvfp4_weights(N, Kin, 1610 + i)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        items.append((outs[src], *_nv_upload(w, dev), y))
        indep.append(name in ("k", "v", "up"))
        outs[name] = y
        ws.append(w)
    chain = aq.Chain(items, group_size=16, bits=4, independent=indep)
    for rep in range(2):
        for it in items:
            it[4].fill_(float("nan"))
        chain.run()
        torch.cuda.synchronize()
        assert aq.aq_read_device_status(None) == aq.AQ_OK
        for i, ((xin, wt, st, gs, y), w) in enumerate(zip(items, ws)):
            scale = float(gs.item())
            Kin = w.K
            xh = from_dev_bf16(xin).reshape(M, Kin)
            _, ref = oracle.nvfp4_matmul(xh, w.w_packed, w.scales, scale, M, w.N, Kin)
            assert_parity(from_dev_bf16(y), ref, what=f"{plan[i][0]} (run {rep})")
            assert torch.equal(y, aq.matmul_nvfp4(xin, wt, st, scale)), plan[i][0]
        # the second run reads new tensor scales from the same device floats
        for it in items:
            it[3].mul_(0.5)


# ---------------------------------------------------------------- release only where memory is shared

def _plan_of(dev, items, independent=None, release=None, group_size=64, bits=4):
    chain = aq.Chain(items, group_size=group_size, bits=bits, independent=independent, release=release)
    return chain, int(chain.plan.reserved[3])


def test_chain_releases_only_where_a_later_matmul_touches_earlier_memory(dev):
    """aq_chain_prepare publishes a group's completion with a GPU-scope release
    only where a later matmul reads or rewrites memory written up to that
    group, or rewrites memory read up to it (the plan reports how many
    groups); results are the same bits either way, and AQ_CHAIN_RELEASE
    forces the release on every group."""
    import torch
    K = 1024
    ws = [synth.make_weights(K, K, 1900 + i) for i in range(4)]
    wdev = [upload(np.zeros((1, K), np.uint16), w, dev)[1:] for w in ws]
    x = to_dev_bf16(synth.make_x(1, K, 1900), dev)
    xs = [to_dev_bf16(synth.make_x(1, K, 1901 + i), dev) for i in range(4)]
    ys = [torch.empty((1, K), dtype=torch.bfloat16, device=dev) for _ in range(4)]

    # separate inputs and outputs (the decode step's layout): ordering only, no release
    items = [(xs[i], *wdev[i], ys[i]) for i in range(4)]
    chain, n = _plan_of(dev, items)
    assert n == 0
    chain.run()
    torch.cuda.synchronize()
    ref = [y.clone() for y in ys]
    for i in range(4):
        assert torch.equal(ys[i], aq.matmul(xs[i], *wdev[i])), i
    # forced: every group but the last (whose completion nothing in the chain awaits)
    chain_f, n_f = _plan_of(dev, items, release=True)
    assert n_f == 3
    for y in ys:
        y.fill_(float("nan"))
    chain_f.run()
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(ys, ref))

    # read after write: matmul 2 reads matmul 0's output -> groups 0 and 1 released
    items_raw = [(x, *wdev[0], ys[0]), (xs[1], *wdev[1], ys[1]), (ys[0], *wdev[2], ys[2]), (xs[3], *wdev[3], ys[3])]
    chain_raw, n_raw = _plan_of(dev, items_raw)
    assert n_raw == 2
    for _ in range(3):
        for y in ys:
            y.fill_(float("nan"))
        chain_raw.run()
        torch.cuda.synchronize()
        y0 = aq.matmul(x, *wdev[0])
        assert torch.equal(ys[0], y0)
        assert torch.equal(ys[2], aq.matmul(y0, *wdev[2]))
    assert aq.aq_read_device_status(None) == aq.AQ_OK

    # write after read: matmul 3 overwrites matmul 1's input -> groups 1 and 2 released
    xw = xs[1].clone()
    items_war = [(xs[0], *wdev[0], ys[0]), (xw, *wdev[1], ys[1]), (xs[2], *wdev[2], ys[2]), (xs[3], *wdev[3], xw)]
    chain_war, n_war = _plan_of(dev, items_war)
    assert n_war == 2
    chain_war.run()
    torch.cuda.synchronize()
    assert torch.equal(ys[1], aq.matmul(xs[1], *wdev[1]))
    assert torch.equal(xw, aq.matmul(xs[3], *wdev[3]))

    # independent matmuls: a hazard between groups still marks every group it crosses
    items_ind = [(x, *wdev[0], ys[0]), (x, *wdev[1], ys[1]), (xs[2], *wdev[2], ys[2]), (ys[1], *wdev[3], ys[3])]
    _, n_ind = _plan_of(dev, items_ind, independent=[False, True, False, False])
    assert n_ind == 2          # groups {0, 1} and {2}
