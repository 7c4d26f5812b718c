"""GPU path (through the C ABI) against the CPU oracle, element by element.

Layout and dispatch must match bit for bit; combine within 1 bf16 ulp (the
tolerance of the fixed-order fp32 reduction; the fma chain is the same on
both sides, so the tests also require bit-exact equality where noted).
Every workload of the benchmark is checked at full size, at the SM budgets
the benchmark uses, plus edge cases (empty, ragged, masked, invalid ids,
maximum K and E, multi-chunk rows).
"""
from __future__ import annotations

import dataclasses
import functools

import numpy as np
import pytest
import torch

import oracle
from combine_movement_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CANARY = 0x7FA5  # a NaN bit pattern no copied row carries


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    from combine_movement_gb300 import build
    build.build()
    yield
    from combine_movement_gb300 import ep
    ep.ep_set_num_sms(0)


@pytest.fixture(scope="module")
def ep():
    from combine_movement_gb300 import ep as mod
    return mod


@functools.lru_cache(maxsize=None)
def _oracle():
    return oracle.Oracle()


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    def ordered(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u)
    return np.abs(ordered(a) - ordered(b))


@dataclasses.dataclass
class Ref:
    counts: np.ndarray
    offsets: np.ndarray
    slot: np.ndarray
    status: int
    recv_x: np.ndarray
    recv_w: np.ndarray
    recv_src: np.ndarray
    expert_out: np.ndarray
    y: np.ndarray


def oracle_path(inp: W.Inputs, num_recv: int, expert_scale: float) -> Ref:
    o = _oracle()
    idx = inp.topk_idx.numpy()
    counts, offsets, slot, st = o.layout(idx, inp.wl.E)
    recv_x, recv_w, recv_src = o.dispatch(inp.x_bits(), slot, num_recv, inp.topk_w.numpy(),
                                          fill=CANARY)
    eo = bits(W.expert_standin(from_bits(recv_x), expert_scale))
    y = o.combine(eo, slot, inp.topk_w.numpy())
    return Ref(counts, offsets, slot, st, recv_x, recv_w, recv_src, eo, y)


def gpu_path(ep, inp: W.Inputs, num_recv: int, expert_out: np.ndarray, num_sms: int = 0,
             stream=None, fused: bool = False, idx_shifted: bool = False):
    dev = torch.device("cuda:0")
    E = inp.wl.E
    ep.ep_set_num_sms(num_sms)
    idx = inp.topk_idx.to(dev)
    if idx_shifted:
        # the same table starting 8 bytes past a 16-byte boundary
        buf = torch.empty(idx.numel() + 1, dtype=torch.int64, device=dev)
        buf[1:] = idx.reshape(-1)
        idx = buf[1:].view(idx.shape)
        assert idx.data_ptr() % 16 == 8
    w = inp.topk_w.to(dev)
    x = inp.x.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    T, K = idx.shape
    counts = torch.full((E,), -7, dtype=torch.int32, device=dev)
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    slot = torch.full((T, K), -7, dtype=torch.int32, device=dev)
    nws = ep.ep_layout_workspace_bytes(T, K, E)
    ws = torch.full((max(nws, 4),), 0x55, dtype=torch.uint8, device=dev) if nws else None
    recv_x = torch.full((num_recv, inp.wl.H), CANARY, dtype=torch.int16,
                        device=dev).view(torch.bfloat16)
    recv_w = torch.full((num_recv,), float("nan"), dtype=torch.float32, device=dev)
    recv_src = torch.full((num_recv,), -1, dtype=torch.int32, device=dev)
    y = torch.full((T, inp.wl.H), 3.0, dtype=torch.bfloat16, device=dev)
    eo = from_bits(expert_out).to(dev)
    if fused:
        ep.ep_layout_dispatch(idx, E, x, counts, offsets, slot, recv_x, w, recv_w, recv_src,
                              status, stream)
    else:
        ep.ep_get_dispatch_layout(idx, E, counts, offsets, slot, ws, status, stream)
        ep.ep_dispatch(x, slot, recv_x, w, recv_w, recv_src, status, stream)
    ep.ep_combine(eo, slot, w, y, status, stream)
    st = ep.ep_get_status(status, stream)
    torch.cuda.synchronize()
    return dict(counts=counts.cpu().numpy(), offsets=offsets.cpu().numpy(),
                slot=slot.cpu().numpy(), recv_x=bits(recv_x), recv_w=recv_w.cpu().numpy(),
                recv_src=recv_src.cpu().numpy(), y=bits(y), status=st)


def assert_parity(got: dict, ref: Ref, exact_combine: bool = True) -> None:
    assert got["status"] == ref.status, (got["status"], ref.status)
    assert np.array_equal(got["counts"], ref.counts), "counts"
    assert np.array_equal(got["offsets"], ref.offsets), "offsets"
    assert np.array_equal(got["slot"], ref.slot), "slot"
    assert np.array_equal(got["recv_x"], ref.recv_x), "recv_x (incl. untouched canary rows)"
    assert np.array_equal(got["recv_w"], ref.recv_w, equal_nan=True), "recv_w"
    assert np.array_equal(got["recv_src"], ref.recv_src), "recv_src"
    d = ulp_distance(got["y"], ref.y)
    assert int(d.max(initial=0)) <= 1, f"combine off by {int(d.max())} ulp"
    if exact_combine:
        assert np.array_equal(got["y"], ref.y), f"combine: {int((d > 0).sum())} elements differ by 1 ulp"


@functools.lru_cache(maxsize=2)
def _case(name: str):
    wl = {"tiny": W.TINY, "decode": W.DECODE, "skewed": W.SKEWED,
          "deepseek": W.DEEPSEEK_PREFILL}.get(name)
    if wl is None:
        T, H = (int(v) for v in name.split(":"))
        wl = W.sweep(T, H)
    inp = W.make_inputs(wl)
    R = wl.T * wl.K
    return inp, oracle_path(inp, R, wl.expert_scale)


@pytest.mark.parametrize("name,budgets", [
    ("tiny", (0, 1, 8)),
    ("decode", (0, 16, 24)),
    ("skewed", (0, 24)),
    ("deepseek", (0, 8, 16, 24, 48)),
])
def test_workloads_full_size(ep, name, budgets):
    inp, ref = _case(name)
    for b in budgets:
        got = gpu_path(ep, inp, inp.wl.T * inp.wl.K, ref.expert_out, num_sms=b)
        assert_parity(got, ref)


@pytest.mark.parametrize("T", W.SWEEP_T)
@pytest.mark.parametrize("H", W.SWEEP_H)
def test_size_sweep(ep, T, H):
    inp, ref = _case(f"{T}:{H}")
    budgets = (0, 8, 16, 24, 48) if T * H <= 4096 * 7168 else (0, 24)
    for b in budgets:
        got = gpu_path(ep, inp, T * 8, ref.expert_out, num_sms=b)
        assert_parity(got, ref)


def _custom(T, H, E, K, seed=7, mask=0.0, routing="uniform"):
    wl = W.Workload(f"edge-T{T}-H{H}-E{E}-K{K}", T=T, H=H, E=E, K=K, seed=seed,
                    mask_frac=mask, routing=routing)
    return W.make_inputs(wl)


@pytest.mark.parametrize("T,H,E,K,mask", [
    (1, 8, 1, 1, 0.0),          # smallest everything; 16-byte rows
    (3, 24, 2, 2, 0.0),         # ragged 48-byte rows (partial column block)
    (33, 520, 5, 3, 0.0),       # odd sizes, T*K not a multiple of 32
    (257, 16384, 16, 4, 0.0),   # multi-chunk rows (32 KB)
    (300, 7176, 64, 8, 0.0),    # H not a multiple of the chunk or 512-byte block
    (500, 1024, 128, 6, 0.3),   # masked entries (-1)
    (64, 256, 4096, 8, 0.0),    # maximum expert count, mostly empty experts
    (2048, 256, 4096, 8, 0.0),  # maximum expert count, one 16-CTA cluster (else cooperative)
    (2100, 256, 4096, 8, 0.0),  # maximum expert count, just past it: cooperative layout
    (40, 64, 40, 32, 0.0),      # maximum K (generic combine path)
    (100, 128, 16, 12, 0.1),    # K above the specialised range, masked
    (9000, 64, 256, 1, 0.0),    # K = 1, multi-tile layout
    (20000, 16, 4096, 8, 0.05), # more tiles than one launch holds: tile + finish kernels
    (70000, 8, 4096, 8, 0.0),   # over 512 tiles: separate one-block scan
    (300, 2048, 16, 5, 0.0),    # K = 5: combine at 1024 threads, row pointers
    (257, 1000, 32, 7, 0.05),   # K = 7: rows by slot index; masked and partial-row units
    (129, 4104, 64, 6, 0.0),    # K = 6: rows by slot index, last unit partial
])
def test_edge_shapes(ep, T, H, E, K, mask):
    inp = _custom(T, H, E, K, mask=mask)
    R_valid = int((inp.topk_idx >= 0).sum())
    num_recv = R_valid + 3  # spare rows must stay untouched
    ref = oracle_path(inp, num_recv, 1.0)
    assert int(ref.offsets[-1]) == R_valid
    for b in (0, 3):
        assert_parity(gpu_path(ep, inp, num_recv, ref.expert_out, num_sms=b), ref)


@pytest.mark.parametrize("K", range(1, 9))
@pytest.mark.parametrize("mask", [0.0, 0.2])
def test_narrow_combine_shapes_every_k(ep, K, mask):
    """Below the wide budgets each K has its own combine shape (threads,
    two or four 512-byte column blocks per unit, row addressing). Rows of
    7184 bytes hold whole units plus a 16-byte tail, so both the unpredicated
    body and the predicated one run, with and without masked entries."""
    inp = _custom(200, 3592, 32, K, seed=40 + K, mask=mask)
    num_recv = int((inp.topk_idx >= 0).sum()) + 2
    ref = oracle_path(inp, num_recv, 1.5)
    for b in (3, 24):
        assert_parity(gpu_path(ep, inp, num_recv, ref.expert_out, num_sms=b), ref)


def _fuzz_cases(n=24, seed=2024):
    """Seeded random shapes: T, H (a multiple of 8), E, K <= min(E, 32),
    masking, routing and SM budget drawn at random, sized so the oracle
    finishes each in well under a second."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        E = int(rng.choice([1, 2, 3, 7, 16, 33, 64, 128, 256, 300, 1024, 4096]))
        K = int(rng.integers(1, min(E, 32) + 1))
        T = int(rng.integers(1, 3000))
        H = 8 * int(rng.integers(1, 1200))
        while T * H > 4_000_000:
            H = max(8, H // 2 // 8 * 8)
            T = max(1, T // 2)
        mask = float(rng.choice([0.0, 0.0, 0.05, 0.5]))
        routing = "zipf" if (rng.random() < 0.3 and K < E) else "uniform"
        budget = int(rng.choice([0, 0, 1, 2, 5, 24, 100]))
        cases.append((T, H, E, K, mask, routing, budget, 100 + i))
    return cases


def _fuzz_small_cases(n=24, seed=4048):
    """Seeded random small tables (at most 4096 routing entries) on partial
    budgets: the shapes that take ep_layout_dispatch's one-launch form, where
    every CTA lays out the table itself before its ring starts."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        E = int(rng.choice([1, 2, 5, 16, 33, 128, 256, 1000, 4096]))
        K = int(rng.integers(1, min(E, 8) + 1))
        T = int(rng.integers(1, 4096 // K + 1))
        H = 8 * int(rng.integers(1, 1025))
        while T * H > 3_000_000:
            T = max(1, T // 2)
        mask = float(rng.choice([0.0, 0.0, 0.1, 0.5]))
        routing = "zipf" if (rng.random() < 0.3 and K < E) else "uniform"
        budget = int(rng.choice([1, 2, 3, 5, 16, 24, 48]))
        cases.append((T, H, E, K, mask, routing, budget, 300 + i))
    return cases


@pytest.mark.parametrize("T,H,E,K,mask,routing,budget,seed", _fuzz_small_cases())
def test_random_small_tables_both_call_forms(ep, T, H, E, K, mask, routing, budget, seed):
    inp = _custom(T, H, E, K, seed=seed, mask=mask, routing=routing)
    num_recv = int((inp.topk_idx >= 0).sum()) + 1
    ref = oracle_path(inp, num_recv, 1.5)
    assert_parity(gpu_path(ep, inp, num_recv, ref.expert_out, num_sms=budget, fused=True), ref)
    assert_parity(gpu_path(ep, inp, num_recv, ref.expert_out, num_sms=budget), ref)


@pytest.mark.parametrize("T,H,E,K,mask,routing,budget,seed", _fuzz_cases())
def test_random_shapes(ep, T, H, E, K, mask, routing, budget, seed):
    inp = _custom(T, H, E, K, seed=seed, mask=mask, routing=routing)
    R_valid = int((inp.topk_idx >= 0).sum())
    num_recv = R_valid + 1
    ref = oracle_path(inp, num_recv, 1.5)
    assert_parity(gpu_path(ep, inp, num_recv, ref.expert_out, num_sms=budget), ref)
    # the same case through ep_layout_dispatch (one or two launches)
    assert_parity(gpu_path(ep, inp, num_recv, ref.expert_out, num_sms=budget, fused=True), ref)


def test_empty_batch(ep):
    inp = _custom(0, 64, 8, 2)
    ref = oracle_path(inp, 0, 1.0)
    got = gpu_path(ep, inp, 0, ref.expert_out)
    assert got["status"] == 0
    assert np.array_equal(got["counts"], np.zeros(8, np.int32))
    assert np.array_equal(got["offsets"], np.zeros(9, np.int32))


def test_hot_expert_and_duplicates(ep):
    # every token sends all K picks to expert 0 or repeats an expert
    T, H, E, K = 1500, 512, 8, 4
    inp = _custom(T, H, E, K)
    idx = inp.topk_idx.clone()
    idx[: T // 2] = 0
    idx[T // 2:, 1] = idx[T // 2:, 0]
    inp = dataclasses.replace(inp, topk_idx=idx.contiguous())
    ref = oracle_path(inp, T * K, 1.0)
    assert int(ref.counts[0]) >= 2 * T  # the hot expert
    for b in (0, 5):
        assert_parity(gpu_path(ep, inp, T * K, ref.expert_out, num_sms=b), ref)


def test_bad_expert_ids_are_skipped_and_reported(ep):
    inp = _custom(700, 64, 32, 4)
    idx = inp.topk_idx.clone()
    idx[5, 1] = 32
    idx[600, 3] = -9
    idx[17, 0] = -1
    inp = dataclasses.replace(inp, topk_idx=idx.contiguous())
    ref = oracle_path(inp, 700 * 4, 1.0)
    assert ref.status == oracle.BAD_EXPERT
    got = gpu_path(ep, inp, 700 * 4, ref.expert_out)
    assert got["status"] == ep.EP_ERR_BAD_EXPERT
    got["status"] = ref.status
    assert_parity(got, ref)


def test_receive_buffer_too_small_is_reported(ep):
    inp = _custom(64, 64, 4, 2)
    ref = oracle_path(inp, 64 * 2, 1.0)
    dev = torch.device("cuda:0")
    slot = torch.from_numpy(ref.slot).to(dev)
    x = inp.x.to(dev)
    small = torch.zeros((100, 64), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ep.ep_set_num_sms(0)
    ep.ep_dispatch(x, slot, small, status=status)
    assert ep.ep_get_status(status) == ep.EP_ERR_BAD_SLOT
    # rows that fit were written
    ok = ref.slot.reshape(-1) < 100
    rows = ref.slot.reshape(-1)[ok]
    assert np.array_equal(bits(small)[rows], ref.recv_x[rows])
    status.zero_()
    y = torch.empty((64, 64), dtype=torch.bfloat16, device=dev)
    ep.ep_combine(small, slot, inp.topk_w.to(dev), y, status=status)
    assert ep.ep_get_status(status) == ep.EP_ERR_BAD_SLOT


def test_combine_closed_forms_on_gpu(ep):
    # all weights 1 with identity experts gives bf16(K*x); one-hot gives x
    T, H, E, K = 512, 7168, 256, 8
    inp = _custom(T, H, E, K)
    dev = torch.device("cuda:0")
    ep.ep_set_num_sms(0)
    counts, offsets, slot = ep.get_dispatch_layout(inp.topk_idx.to(dev), E)
    x = inp.x.to(dev)
    recv = ep.dispatch(x, slot, T * K)
    ones = torch.ones((T, K), dtype=torch.float32, device=dev)
    y = ep.combine(recv, slot, ones)
    want = (inp.x.float() * K).to(torch.bfloat16)
    assert np.array_equal(bits(y), bits(want))
    oh = torch.zeros((T, K), dtype=torch.float32, device=dev)
    oh[:, K - 1] = 1.0
    assert np.array_equal(bits(ep.combine(recv, slot, oh)), bits(inp.x))


def test_side_stream_and_repeat_determinism(ep):
    inp, ref = _case("skewed")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = gpu_path(ep, inp, inp.wl.T * inp.wl.K, ref.expert_out, num_sms=24, stream=s)
    b = gpu_path(ep, inp, inp.wl.T * inp.wl.K, ref.expert_out, num_sms=24)
    assert_parity(a, ref)
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True)


def test_back_to_back_batches_share_buffers_on_one_stream(ep):
    """Several batches through the same device buffers on one stream with no
    host synchronisation between them. Every kernel is launched with
    programmatic dependent launch and may start while the previous one
    finishes, so this checks that each still sees its producer's writes
    (slot, recv_x, the expert stand-in's output) and that no kernel of a
    batch overwrites what a kernel of the previous batch still reads."""
    dev = torch.device("cuda:0")
    T, H, E, K = 1536, 1032, 64, 6
    cases = [(11, "uniform", 0.0, 1.5), (12, "zipf", 0.1, 1.0),
             (13, "uniform", 0.2, 1.5), (14, "zipf", 0.0, 1.0)]
    inps = [_custom(T, H, E, K, seed=sd, mask=m, routing=r) for sd, r, m, _ in cases]
    refs = [oracle_path(inp, T * K, sc) for inp, (_, _, _, sc) in zip(inps, cases)]
    idx = [inp.topk_idx.to(dev) for inp in inps]
    w = [inp.topk_w.to(dev) for inp in inps]
    x = [inp.x.to(dev) for inp in inps]
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    slot = torch.empty((T, K), dtype=torch.int32, device=dev)
    nws = ep.ep_layout_workspace_bytes(T, K, E)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev) if nws else None
    recv = torch.empty((T * K, H), dtype=torch.bfloat16, device=dev)
    eo = torch.empty((T * K, H), dtype=torch.bfloat16, device=dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = [dict(slot=torch.empty((T, K), dtype=torch.int32).pin_memory(),
                offsets=torch.empty(E + 1, dtype=torch.int32).pin_memory(),
                recv=torch.empty((T * K, H), dtype=torch.bfloat16).pin_memory(),
                y=torch.empty((T, H), dtype=torch.bfloat16).pin_memory()) for _ in cases]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    # budgets with the default launch policy, 24 SMs with overlapping
    # launches forced on, and the full budget with them forced off (each
    # combination also changes the dispatch ring: 3 stages while launches
    # overlap, else 4)
    for b, mode in ((0, 0), (24, 0), (24, 1), (0, 2)):
        ep.ep_set_num_sms(b)
        ep.ep_set_launch_overlap(mode)
        with torch.cuda.stream(s):
            for i, (_, _, _, sc) in enumerate(cases):
                ep.ep_get_dispatch_layout(idx[i], E, counts, offsets, slot, ws, status, s)
                ep.ep_dispatch(x[i], slot, recv, None, None, None, status, s)
                eo.copy_(W.expert_standin(recv, sc))
                ep.ep_combine(eo, slot, w[i], y, status, s)
                for name, src in (("slot", slot), ("offsets", offsets), ("recv", recv), ("y", y)):
                    out[i][name].copy_(src, non_blocking=True)
        s.synchronize()
        assert ep.ep_get_status(status) == ep.EP_OK
        for i, ref in enumerate(refs):
            assert np.array_equal(out[i]["slot"].numpy(), ref.slot), f"batch {i}: slot"
            assert np.array_equal(out[i]["offsets"].numpy(), ref.offsets), f"batch {i}: offsets"
            r = bits(out[i]["recv"])
            valid = int(ref.offsets[-1])
            assert np.array_equal(r[:valid], ref.recv_x[:valid]), f"batch {i}: recv_x"
            assert np.array_equal(bits(out[i]["y"]), ref.y), f"batch {i}: y"
    ep.ep_set_num_sms(0)
    ep.ep_set_launch_overlap(0)


def test_layers_chained_through_layout_dispatch_on_one_stream(ep):
    """Four MoE layers back to back on one stream with no host
    synchronisation, each layer's combine output being the next layer's
    input x (as in a model), through ep_layout_dispatch + ep_combine. With
    launch overlap, a dispatch whose layout kernel precedes it issues its
    first row loads before waiting for that kernel; x is then the previous
    layer's combine output, complete only because the layout kernel waits
    for it before it lets dispatch launch. Every layer's slots, rows and
    output are compared with the oracle's chain, at the full budget (launch
    overlap on), at 24 SMs (off) and at 24 SMs with it forced on."""
    dev = torch.device("cuda:0")
    T, H = 300, 2056
    layers = [(64, 6, "uniform", 1.5), (256, 8, "zipf", 1.0), (16, 2, "uniform", 1.5),
              (128, 1, "uniform", 1.0)]
    first = _custom(T, H, layers[0][0], layers[0][1], seed=70)
    routes = [_custom(T, 8, E, K, seed=71 + i, routing=r) for i, (E, K, r, _) in enumerate(layers)]
    # the oracle's chain
    x_bits = first.x_bits()
    refs = []
    for (E, K, _, sc), rt in zip(layers, routes):
        o = _oracle()
        counts, offsets, slot, st = o.layout(rt.topk_idx.numpy(), E)
        recv_x, _, _ = o.dispatch(x_bits, slot, T * K, rt.topk_w.numpy(), fill=CANARY)
        eo = bits(W.expert_standin(from_bits(recv_x), sc))
        y = o.combine(eo, slot, rt.topk_w.numpy())
        refs.append((slot, recv_x, y))
        x_bits = y
    s = torch.cuda.Stream()
    try:
        for b, mode in ((0, 0), (24, 0), (24, 1)):
            ep.ep_set_num_sms(b)
            ep.ep_set_launch_overlap(mode)
            with torch.cuda.stream(s):
                x = first.x.to(dev)
                status = torch.zeros(1, dtype=torch.int32, device=dev)
                outs = []
                for (E, K, _, sc), rt in zip(layers, routes):
                    idx, w = rt.topk_idx.to(dev), rt.topk_w.to(dev)
                    counts = torch.empty(E, dtype=torch.int32, device=dev)
                    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
                    slot = torch.full((T, K), -5, dtype=torch.int32, device=dev)
                    recv = torch.empty((T * K, H), dtype=torch.bfloat16, device=dev)
                    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
                    ep.ep_layout_dispatch(idx, E, x, counts, offsets, slot, recv, None, None, None,
                                          status, s)
                    eo = W.expert_standin(recv, sc)
                    ep.ep_combine(eo, slot, w, y, status, s)
                    outs.append((slot, recv, y))
                    x = y
            s.synchronize()
            assert ep.ep_get_status(status) == ep.EP_OK
            for i, ((slot, recv, y), (r_slot, r_recv, r_y)) in enumerate(zip(outs, refs)):
                assert np.array_equal(slot.cpu().numpy(), r_slot), f"budget {b}, mode {mode}, layer {i}: slot"
                assert np.array_equal(bits(recv), r_recv), f"budget {b}, mode {mode}, layer {i}: recv_x"
                assert np.array_equal(bits(y), r_y), f"budget {b}, mode {mode}, layer {i}: y"
    finally:
        ep.ep_set_num_sms(0)
        ep.ep_set_launch_overlap(0)


def _stream_mix(n=12, seed=5151):
    """Seeded heterogeneous batches: any table size up to 24K entries (every
    layout launch shape but the largest), any row size, either call form."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.choice([1, 8, 64, 256, 1024, 4096]))
        K = int(rng.integers(1, min(E, 8) + 1))
        T = int(rng.integers(1, 3000))
        H = 8 * int(rng.integers(1, 600))
        mask = float(rng.choice([0.0, 0.0, 0.2]))
        out.append((T, H, E, K, mask, bool(rng.random() < 0.5), 500 + i))
    return out


@functools.lru_cache(maxsize=1)
def _stream_mix_inputs():
    """Inputs and oracle results of _stream_mix(), computed once."""
    res = []
    for T, H, E, K, mask, fused, seed in _stream_mix():
        inp = _custom(T, H, E, K, seed=seed, mask=mask)
        num_recv = int((inp.topk_idx >= 0).sum()) + 1
        res.append((inp, num_recv, oracle_path(inp, num_recv, 1.0)))
    return res


@pytest.mark.parametrize("budget,mode", [(0, 0), (24, 1), (5, 0)])
def test_heterogeneous_batches_back_to_back(ep, budget, mode):
    """Twelve unrelated batches (random sizes, layout launch shapes and call
    forms, each with its own buffers) issued back to back on one stream with
    no host synchronisation, with launch overlap (the default at the full
    budget, forced at 24 SMs) and without it (5 SMs): each kernel may start
    while a kernel of another shape finishes."""
    dev = torch.device("cuda:0")
    cases = _stream_mix()
    prepared = _stream_mix_inputs()
    refs, runs = [], []
    s = torch.cuda.Stream()
    try:
        ep.ep_set_num_sms(budget)
        ep.ep_set_launch_overlap(mode)
        for (T, H, E, K, mask, fused, seed), (inp, num_recv, ref) in zip(cases, prepared):
            refs.append(ref)
            with torch.cuda.stream(s):
                idx, w, x = inp.topk_idx.to(dev), inp.topk_w.to(dev), inp.x.to(dev)
                counts = torch.empty(E, dtype=torch.int32, device=dev)
                offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
                slot = torch.empty((T, K), dtype=torch.int32, device=dev)
                recv = torch.full((num_recv, H), CANARY, dtype=torch.int16,
                                  device=dev).view(torch.bfloat16)
                y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
                status = torch.zeros(1, dtype=torch.int32, device=dev)
                if fused:
                    ep.ep_layout_dispatch(idx, E, x, counts, offsets, slot, recv, None, None,
                                          None, status, s)
                else:
                    nws = ep.ep_layout_workspace_bytes(T, K, E)
                    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev) if nws else None
                    ep.ep_get_dispatch_layout(idx, E, counts, offsets, slot, ws, status, s)
                    ep.ep_dispatch(x, slot, recv, None, None, None, status, s)
                ep.ep_combine(recv, slot, w, y, status, s)
                runs.append((counts, offsets, slot, recv, y, status, ws if not fused else None))
        s.synchronize()
        for (T, H, E, K, mask, fused, seed), ref, (counts, offsets, slot, recv, y, status, _) in zip(
                cases, refs, runs):
            what = f"T={T} H={H} E={E} K={K} fused={fused}"
            assert ep.ep_get_status(status) == ep.EP_OK, what
            assert np.array_equal(counts.cpu().numpy(), ref.counts), what
            assert np.array_equal(offsets.cpu().numpy(), ref.offsets), what
            assert np.array_equal(slot.cpu().numpy(), ref.slot), what
            assert np.array_equal(bits(recv), ref.recv_x), what
            assert np.array_equal(bits(y), ref.y), what
    finally:
        ep.ep_set_num_sms(0)
        ep.ep_set_launch_overlap(0)


@pytest.mark.parametrize("T,H,E,K", [
    (128, 7168, 256, 8),   # decode: one-block layout
    (2048, 2048, 64, 8),   # one thread-block cluster layout
    (16384, 64, 128, 8),   # one 16-CTA cluster (where the GPU holds one; else cooperative)
    (20000, 64, 128, 8),   # cooperative layout (grid barrier, generation word)
])
def test_cuda_graph_capture_and_replay(ep, T, H, E, K):
    """The three calls captured once into a CUDA graph (with the expert
    stand-in between them) and replayed on new inputs copied into the same
    buffers: every entry point only enqueues launches, so the graph replays
    the whole step; each replay is compared with the oracle."""
    dev = torch.device("cuda:0")
    inps = [_custom(T, H, E, K, seed=20 + i) for i in range(3)]
    refs = [oracle_path(inp, T * K, 1.5) for inp in inps]
    idx = inps[0].topk_idx.to(dev).clone()
    w = inps[0].topk_w.to(dev).clone()
    x = inps[0].x.to(dev).clone()
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    slot = torch.empty((T, K), dtype=torch.int32, device=dev)
    nws = ep.ep_layout_workspace_bytes(T, K, E)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev) if nws else None
    recv = torch.empty((T * K, H), dtype=torch.bfloat16, device=dev)
    eo = torch.empty((T * K, H), dtype=torch.bfloat16, device=dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ep.ep_set_num_sms(24)

    def step(stream):
        ep.ep_get_dispatch_layout(idx, E, counts, offsets, slot, ws, status, stream)
        ep.ep_dispatch(x, slot, recv, None, None, None, status, stream)
        eo.copy_(W.expert_standin(recv, 1.5))
        ep.ep_combine(eo, slot, w, y, status, stream)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(s)  # eager warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream())
    try:
        for inp, ref in zip(inps, refs):
            idx.copy_(inp.topk_idx)
            w.copy_(inp.topk_w)
            x.copy_(inp.x)
            slot.fill_(-9)
            y.fill_(0)
            g.replay()
            torch.cuda.synchronize()
            assert ep.ep_get_status(status) == ep.EP_OK
            assert np.array_equal(slot.cpu().numpy(), ref.slot)
            assert np.array_equal(offsets.cpu().numpy(), ref.offsets)
            assert np.array_equal(bits(y), ref.y)
    finally:
        ep.ep_set_num_sms(0)


# ---- ep_layout_dispatch: layout and dispatch in one call (one or two launches)

@pytest.mark.parametrize("name,budgets", [
    ("tiny", (0, 3)),
    ("decode", (0, 16, 24)),
    ("skewed", (0, 24)),
    ("deepseek", (0, 8, 24)),
])
def test_fused_layout_dispatch_workloads(ep, name, budgets):
    inp, ref = _case(name)
    for b in budgets:
        got = gpu_path(ep, inp, inp.wl.T * inp.wl.K, ref.expert_out, num_sms=b, fused=True)
        assert_parity(got, ref)


@pytest.mark.parametrize("T,H,E,K,mask", [
    (0, 64, 8, 2, 0.0),
    (1, 8, 1, 1, 0.0),
    (3, 24, 2, 2, 0.0),
    (257, 16384, 16, 4, 0.0),
    (500, 1024, 128, 6, 0.3),
    (64, 256, 4096, 8, 0.0),
    (40, 64, 40, 32, 0.0),
    (2000, 64, 256, 1, 0.1),
])
def test_fused_layout_dispatch_edges(ep, T, H, E, K, mask):
    inp = _custom(T, H, E, K, mask=mask)
    R_valid = int((inp.topk_idx >= 0).sum())
    ref = oracle_path(inp, R_valid + 3, 1.0)
    for b in (0, 5):
        assert_parity(gpu_path(ep, inp, R_valid + 3, ref.expert_out, num_sms=b, fused=True), ref)


@pytest.mark.parametrize("T,H,E,K,budget", [
    (150, 3096, 128, 1, 1),   # 75 id pairs: warp 2 split by the id count, rows to move; 205 KB of shared memory
    (150, 3096, 128, 1, 2),
    (91, 6200, 64, 2, 1),     # 91 pairs: warp 2 split
    (77, 5600, 33, 3, 1),     # odd entry count: the last id read on its own
    (300, 1032, 256, 1, 3),   # 150 pairs: warp 4 split
    (40, 7168, 16, 5, 1),     # 100 pairs: warp 3 split; two chunks per row
])
def test_fused_one_launch_warps_split_by_the_id_count(ep, T, H, E, K, budget):
    """The one-launch ep_layout_dispatch (small tables on a partial budget)
    with fewer 16-byte id pairs than threads, not a multiple of 32: one
    warp's lanes straddle the end of the table while the warp also has
    rows to move, and the CTA keeps its entries in shared memory."""
    inp = _custom(T, H, E, K, seed=T + H)
    num_recv = T * K + 1
    ref = oracle_path(inp, num_recv, 1.5)
    assert_parity(gpu_path(ep, inp, num_recv, ref.expert_out, num_sms=budget, fused=True), ref)


@pytest.mark.parametrize("T,H,E,K,mask,routing,short", [
    (16384, 7168, 256, 2, 0.1, "uniform", 0),   # K = 2, masked
    (6144, 7176, 64, 3, 0.0, "uniform", 0),     # 14352-byte rows (a ragged last chunk)
    (2100, 6144, 32, 8, 0.25, "zipf", 0),       # just over the size limit (206 MB)
    (4096, 7168, 256, 8, 0.0, "uniform", 100),  # receive buffer 100 rows short
    (2048, 7168, 64, 12, 0.1, "uniform", 0),    # K = 12: the generic combine path's tail
])
def test_dispatch_tail_launch(ep, T, H, E, K, mask, routing, short):
    """At the full budget, with launches overlapping, a dispatch of at least
    192 MB of receive rows is two launches: a persistent ring over the first
    70 % of the (token, chunk) units, then a tail of small CTAs over the rest
    that start on SMs whose ring CTA has finished; combine splits the same
    way, K above 8 (its generic path) included. Every row must come out
    as the oracle's, through ep_dispatch and ep_layout_dispatch, with masked
    entries, skewed routing, a ragged last chunk, an odd number of tail
    units and rows beyond the receive buffer (reported, not written)."""
    inp = _custom(T, H, E, K, seed=T + K, mask=mask, routing=routing)
    R_valid = int((inp.topk_idx >= 0).sum())
    ref = oracle_path(inp, R_valid, 1.0)   # the oracle gets room for every row
    num_recv = R_valid - short
    ep.ep_set_num_sms(0)
    assert ep.ep_dispatch_launches(T, H, K) == 2
    assert ep.ep_combine_launches(T, H, K) == 2
    for fused in (False, True):
        got = gpu_path(ep, inp, num_recv, ref.expert_out, num_sms=0, fused=fused)
        if short:
            assert got["status"] == ep.EP_ERR_BAD_SLOT
            flat = ref.slot.reshape(-1)
            rows = flat[(flat >= 0) & (flat < num_recv)]
            assert np.array_equal(got["slot"], ref.slot)
            assert np.array_equal(got["recv_x"][rows], ref.recv_x[rows])
        else:
            assert_parity(got, ref)


@functools.lru_cache(maxsize=1)
def _tail_share_case():
    inp = _custom(16384, 7168, 256, 2, seed=911, mask=0.05, routing="zipf")
    R_valid = int((inp.topk_idx >= 0).sum())
    return inp, R_valid, oracle_path(inp, R_valid, 1.5)


@pytest.mark.parametrize("percent", [1, 50, 90])
def test_tail_shares_across_their_range(ep, percent):
    """ep_set_dispatch_tail / ep_set_combine_tail move the split between the
    persistent launch and the tail anywhere in 0-90 %: a tail of a few units,
    one as large as the persistent part, and one nine times larger (the
    persistent ring still keeps two units per warp at this size). Both calls
    stay two launches and every output equals the oracle's, through both
    call forms."""
    inp, R_valid, ref = _tail_share_case()
    T, H, K = inp.wl.T, inp.wl.H, inp.wl.K
    ep.ep_set_num_sms(0)
    try:
        assert ep.ep_set_dispatch_tail(percent) == percent
        assert ep.ep_set_combine_tail(percent) == percent
        assert ep.ep_dispatch_launches(T, H, K) == 2
        assert ep.ep_combine_launches(T, H, K) == 2
        for fused in (False, True):
            assert_parity(gpu_path(ep, inp, R_valid, ref.expert_out, num_sms=0, fused=fused), ref)
    finally:
        ep.ep_set_dispatch_tail(30)
        ep.ep_set_combine_tail(30)


@pytest.mark.parametrize("graph", [False, True])
def test_combine_reads_the_rows_of_both_dispatch_launches(ep, graph):
    """Combine launched right after a two-launch dispatch (ring + tail, the
    whole GPU, launches overlapping) and reading the receive rows
    themselves: it must find the rows of both launches, which holds because
    the tail launch completes after the ring (its last CTA waits for it), so
    combine's wait for its predecessor covers both. Eagerly and replayed
    from a CUDA graph (the programmatic launches captured as such)."""
    T, H, E, K = 2100, 6144, 32, 8
    inps = [_custom(T, H, E, K, seed=60 + i) for i in range(2)]
    refs = [oracle_path(inp, T * K, 1.0) for inp in inps]   # stand-in x1.0: the rows themselves
    dev = torch.device("cuda:0")
    ep.ep_set_num_sms(0)
    assert ep.ep_dispatch_launches(T, H, K) == 2
    idx = inps[0].topk_idx.to(dev).clone()
    w = inps[0].topk_w.to(dev).clone()
    x = inps[0].x.to(dev).clone()
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    slot = torch.empty((T, K), dtype=torch.int32, device=dev)
    recv = torch.empty((T * K, H), dtype=torch.bfloat16, device=dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(stream):
        ep.ep_layout_dispatch(idx, E, x, counts, offsets, slot, recv, None, None, None,
                              status, stream)
        ep.ep_combine(recv, slot, w, y, status, stream)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(s)
    torch.cuda.synchronize()
    g = None
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(torch.cuda.current_stream())
    for inp, ref in zip(inps, refs):
        idx.copy_(inp.topk_idx)
        w.copy_(inp.topk_w)
        x.copy_(inp.x)
        recv.fill_(0)
        y.fill_(0)
        torch.cuda.synchronize()
        if g is not None:
            g.replay()
        else:
            with torch.cuda.stream(s):
                step(s)
        torch.cuda.synchronize()
        assert ep.ep_get_status(status) == ep.EP_OK
        assert np.array_equal(slot.cpu().numpy(), ref.slot)
        assert np.array_equal(bits(recv), ref.recv_x)
        assert np.array_equal(bits(y), ref.y)


def test_two_streams_dispatch_with_tails_at_once(ep):
    """Two independent calls of ep_layout_dispatch + ep_combine, each large
    enough for dispatch's tail launch, issued on two streams with nothing
    ordering them: each tail's last CTA waits only for its own ring, and
    both calls must match the oracle."""
    T, H, E, K = 2100, 6144, 32, 8
    dev = torch.device("cuda:0")
    ep.ep_set_num_sms(0)
    assert ep.ep_dispatch_launches(T, H, K) == 2
    inps = [_custom(T, H, E, K, seed=90 + i, routing=r) for i, r in enumerate(("uniform", "zipf"))]
    refs = [oracle_path(inp, T * K, 1.0) for inp in inps]
    bufs = []
    for inp in inps:
        bufs.append(dict(idx=inp.topk_idx.to(dev), w=inp.topk_w.to(dev), x=inp.x.to(dev),
                         counts=torch.empty(E, dtype=torch.int32, device=dev),
                         offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                         slot=torch.empty((T, K), dtype=torch.int32, device=dev),
                         recv=torch.zeros((T * K, H), dtype=torch.bfloat16, device=dev),
                         y=torch.zeros((T, H), dtype=torch.bfloat16, device=dev),
                         status=torch.zeros(1, dtype=torch.int32, device=dev)))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(3):
        for b, s in zip(bufs, streams):
            with torch.cuda.stream(s):
                ep.ep_layout_dispatch(b["idx"], E, b["x"], b["counts"], b["offsets"], b["slot"],
                                      b["recv"], None, None, None, b["status"], s)
                ep.ep_combine(b["recv"], b["slot"], b["w"], b["y"], b["status"], s)
    torch.cuda.synchronize()
    for b, ref in zip(bufs, refs):
        assert ep.ep_get_status(b["status"]) == ep.EP_OK
        assert np.array_equal(b["slot"].cpu().numpy(), ref.slot)
        assert np.array_equal(bits(b["recv"]), ref.recv_x)
        assert np.array_equal(bits(b["y"]), ref.y)


@pytest.mark.parametrize("T,H,E,K,mask,budget", [
    (16384, 64, 128, 8, 0.0, 0),    # 131,072 entries: 16 tiles of 8 rounds, the most it takes
    (9000, 32, 256, 8, 0.1, 0),     # 72,000 entries: 15 tiles of 5 rounds, masked
    (8200, 8, 33, 8, 0.0, 24),      # 65,600 entries, just past one 8-CTA cluster; partial budget
    (4100, 16, 64, 16, 0.05, 0),    # K = 16
])
def test_layout_dispatch_wide_cluster(ep, T, H, E, K, mask, budget):
    """Tables just past what one 8-CTA cluster lays out (65,536 entries at
    E <= 256) would need a workspace; ep_layout_dispatch, which has none,
    lays them out with one 16-CTA cluster (a non-portable cluster size) and
    keeps its two-launch form. Slots, rows and combine against the oracle,
    and the same results through the three separate calls (whose layout
    keeps its workspace)."""
    inp = _custom(T, H, E, K, seed=T + E, mask=mask)
    R_valid = int((inp.topk_idx >= 0).sum())
    ref = oracle_path(inp, R_valid, 1.0)
    assert ep.ep_layout_workspace_bytes(T, K, E) > 0
    ep.ep_set_num_sms(budget)
    try:
        assert ep.ep_layout_dispatch_launches(T, H, K, E) >= 2   # the layout kernel, then dispatch
    finally:
        ep.ep_set_num_sms(0)
    for fused in (True, False):
        assert_parity(gpu_path(ep, inp, R_valid, ref.expert_out, num_sms=budget, fused=fused), ref)


def test_dispatch_launch_counts(ep):
    """One launch wherever the tail does not apply: decode-size batches, a
    partial SM budget, launch overlap switched off."""
    ep.ep_set_num_sms(0)
    assert ep.ep_dispatch_launches(4096, 7168, 8) == 2
    assert ep.ep_dispatch_launches(128, 7168, 8) == 1
    assert ep.ep_dispatch_launches(1024, 7168, 8) == 1     # 117 MB of rows
    assert ep.ep_dispatch_launches(16384, 7168, 1) == 1    # K = 1
    assert ep.ep_layout_dispatch_launches(4096, 7168, 8, 256) == 3   # layout, ring, tail
    assert ep.ep_layout_dispatch_launches(128, 7168, 8, 256) == 2    # layout, dispatch
    assert ep.ep_combine_launches(4096, 7168, 8) == 2                # persistent, tail
    assert ep.ep_combine_launches(128, 7168, 8) == 1
    mode = ep.ep_get_launch_overlap()
    try:
        ep.ep_set_launch_overlap(2)
        assert ep.ep_dispatch_launches(4096, 7168, 8) == 1
        assert ep.ep_combine_launches(4096, 7168, 8) == 1
    finally:
        ep.ep_set_launch_overlap(mode)
    try:
        ep.ep_set_num_sms(24)
        assert ep.ep_dispatch_launches(4096, 7168, 8) == 1
        assert ep.ep_layout_dispatch_launches(128, 7168, 8, 256) == 1    # one launch
        assert ep.ep_layout_dispatch_launches(4096, 7168, 8, 256) == 2   # more than 4096 entries
    finally:
        ep.ep_set_num_sms(0)


@pytest.mark.parametrize("T,H,E,K,budget,mask,bad,shifted", [
    (128, 256, 128, 8, 8, 0.0, False, False),   # 1024 entries, 128 per CTA, kept in shared memory
    (128, 7168, 575, 8, 24, 0.05, True, False), # decode-size table, three-chunk rows, odd E
    (256, 64, 256, 4, 24, 0.1, True, True),     # masked and out-of-range ids, shifted table
    (205, 64, 256, 5, 24, 0.1, True, True),     # 1025 entries
    (7, 40, 5, 3, 2, 0.0, True, True),          # 21 entries: first id read on its own
    (11, 40, 5, 2, 2, 0.0, False, True),        # first id and odd last id read on their own
    (1, 8, 1, 1, 1, 0.0, False, False),         # one entry
    (100, 512, 4096, 8, 16, 0.05, True, False), # 4096 experts, the last one's id
])
def test_fused_one_launch_edges(ep, T, H, E, K, budget, mask, bad, shifted):
    """The one-launch ep_layout_dispatch (small tables on a partial budget:
    every CTA lays out the whole table before its ring): tables of 1 to
    1025 entries, with masked entries, out-of-range ids, the last expert's
    id, and an id table that starts 8 bytes past a 16-byte boundary (its
    first id then read on its own)."""
    inp = _custom(T, H, E, K, seed=T * 31 + budget, mask=mask)
    idx = inp.topk_idx.clone()
    idx[0, 0] = E - 1
    if bad and T >= 3:
        idx[1, 0] = E + 3
        idx[2, K - 1] = -9
    inp = dataclasses.replace(inp, topk_idx=idx.contiguous())
    num_recv = T * K + 2
    ref = oracle_path(inp, num_recv, 1.25)
    got = gpu_path(ep, inp, num_recv, ref.expert_out, num_sms=budget, fused=True,
                   idx_shifted=shifted)
    if bad and T >= 3:
        assert got["status"] == ep.EP_ERR_BAD_EXPERT
    assert_parity(got, ref)
    if shifted:  # the layout kernel reads the shifted table too
        assert_parity(gpu_path(ep, inp, num_recv, ref.expert_out, num_sms=budget,
                               idx_shifted=True), ref)


@pytest.mark.parametrize("budget", [0, 3])
def test_fused_layout_dispatch_bad_ids(ep, budget):
    # budget 0: the layout kernel and dispatch (launches overlap); 3 SMs:
    # the one-launch form
    inp = _custom(300, 64, 32, 4)
    idx = inp.topk_idx.clone()
    idx[5, 1] = 99
    idx[200, 0] = -4
    inp = dataclasses.replace(inp, topk_idx=idx.contiguous())
    ref = oracle_path(inp, 300 * 4, 1.0)
    got = gpu_path(ep, inp, 300 * 4, ref.expert_out, num_sms=budget, fused=True)
    assert got["status"] == ep.EP_ERR_BAD_EXPERT
    assert_parity(got, ref)


@pytest.mark.parametrize("budget", [0, 3])
def test_fused_layout_dispatch_receive_buffer_too_small(ep, budget):
    """ep_layout_dispatch into a receive buffer of 100 rows for 128
    entries: the rows that fit are written, the others reported."""
    inp = _custom(64, 64, 4, 2)
    ref = oracle_path(inp, 64 * 2, 1.0)
    dev = torch.device("cuda:0")
    ep.ep_set_num_sms(budget)
    try:
        counts = torch.empty(4, dtype=torch.int32, device=dev)
        offsets = torch.empty(5, dtype=torch.int32, device=dev)
        slot = torch.empty((64, 2), dtype=torch.int32, device=dev)
        small = torch.zeros((100, 64), dtype=torch.bfloat16, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        ep.ep_layout_dispatch(inp.topk_idx.to(dev), 4, inp.x.to(dev), counts, offsets, slot, small,
                              status=status)
        assert ep.ep_get_status(status) == ep.EP_ERR_BAD_SLOT
        assert np.array_equal(slot.cpu().numpy(), ref.slot)
        ok = ref.slot.reshape(-1) < 100
        rows = ref.slot.reshape(-1)[ok]
        assert np.array_equal(bits(small)[rows], ref.recv_x[rows])
    finally:
        ep.ep_set_num_sms(0)
