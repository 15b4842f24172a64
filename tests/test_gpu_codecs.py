"""Exhaustive device checks of the producer's building blocks against the
oracle: the BF16 silu over all 65,536 gates, the SwiGLU product, and the
E2M1 / E4M3 encoders over every finite binary32 bit pattern."""
import numpy as np
import pytest
import torch

import oracle
import synth
from diffusion_transformer_mlp_gb300 import _lib

pytestmark = pytest.mark.gpu


def _stream():
    import ctypes
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _p(t):
    import ctypes
    return ctypes.c_void_p(t.data_ptr())


def test_device_silu_all_65536_gates_equal_oracle():
    out = torch.empty(65536, dtype=torch.int16, device="cuda")
    _lib.check(_lib.load().nvfp4_diag_silu_all(_p(out), _stream()), "silu")
    dev = out.cpu().numpy().view(np.uint16)
    ref, unresolved = oracle.silu_table()
    assert unresolved == 0
    gf = synth.bf16_to_f32(np.arange(65536, dtype=np.uint32).astype(np.uint16))
    rf = synth.bf16_to_f32(ref)
    both_nan = np.isnan(synth.bf16_to_f32(dev)) & np.isnan(rf)
    bad = np.nonzero((dev != ref) & ~both_nan)[0]
    assert bad.size == 0, [(hex(i), float(gf[i]), hex(dev[i]), hex(ref[i])) for i in bad[:10]]


def test_device_swiglu_equals_oracle():
    rng = np.random.default_rng(7)
    n = 1 << 18
    g = rng.integers(0, 65536, n).astype(np.uint16)
    u = rng.integers(0, 65536, n).astype(np.uint16)
    # plus the N(0,1) region densely
    g[: n // 2] = synth.normal_bf16((n // 2,), 5, 0, 1.0, 1e-3)
    u[: n // 2] = synth.normal_bf16((n // 2,), 5, 1, 1.0, 1e-3)
    tg = torch.from_numpy(g.view(np.int16)).cuda()
    tu = torch.from_numpy(u.view(np.int16)).cuda()
    th = torch.empty_like(tg)
    _lib.check(_lib.load().nvfp4_diag_swiglu(_p(tg), _p(tu), _p(th), n, _stream()), "swiglu")
    dev = th.cpu().numpy().view(np.uint16)
    tab, _ = oracle.silu_table()
    ref = np.array([oracle.swiglu_bf16(int(a), int(b)) for a, b in zip(g[:20000], u[:20000])], dtype=np.uint16)
    fin = ~np.isnan(synth.bf16_to_f32(ref))
    assert np.array_equal(dev[:20000][fin], ref[fin])
    assert np.all(np.isnan(synth.bf16_to_f32(dev[:20000][~fin])))


def _oracle_transitions(which: int):
    """Transitions of the oracle encoder over the ordered bit patterns, found
    by bisection (the encoders are monotone in |x| within each sign)."""
    enc = oracle.e2m1_encode if which == 0 else oracle.e4m3_encode

    def code(bits):
        return enc(float(np.uint32(bits).view(np.float32)))

    out = []
    for lo, hi in ((0x00000000, 0x7F7FFFFF), (0x80000000, 0xFF7FFFFF)):
        p = lo + 1
        cur = code(lo)
        while p <= hi:
            # first pattern in [p, hi] whose code differs from cur
            if code(hi) == cur:
                break
            a, b = p, hi
            while a < b:
                mid = (a + b) // 2
                if code(mid) != cur:
                    b = mid
                else:
                    a = mid + 1
            new = code(a)
            out.append((a, new, cur))
            cur = new
            p = a + 1
    return sorted(out)


@pytest.mark.parametrize("which", [0, 1], ids=["e2m1", "e4m3"])
def test_device_encoder_transitions_equal_oracle(which):
    cap = 4096
    trans = torch.zeros(3 * cap, dtype=torch.int32, device="cuda")
    count = torch.zeros(1, dtype=torch.int32, device="cuda")
    first = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.check(_lib.load().nvfp4_diag_code_transitions(which, _p(trans), cap, _p(count), _p(first), _stream()),
               "transitions")
    n = int(count.item())
    assert 0 < n <= cap
    t = trans[: 3 * n].cpu().numpy().view(np.uint32).reshape(n, 3)
    dev = sorted(tuple(int(v) for v in row) for row in t)
    ref = _oracle_transitions(which)
    assert int(first.item()) == (oracle.e2m1_encode(0.0) if which == 0 else oracle.e4m3_encode(0.0))
    assert dev == ref, (len(dev), len(ref), [x for x in dev if x not in ref][:5], [x for x in ref if x not in dev][:5])


def test_bounded_wait_reports_timeout_without_hanging():
    st = torch.full((1,), 77, dtype=torch.int32, device="cuda")
    _lib.check(_lib.load().nvfp4_diag_wait_timeout(2_000_000, _p(st), _stream()), "wait")
    torch.cuda.synchronize()
    assert int(st.item()) == _lib.NVFP4_ETIMEOUT
    # the context is still usable
    x = torch.ones(4, device="cuda")
    assert float((x + 1).sum().item()) == 8.0


def test_fp4_mma_loop_runs_and_scales():
    """The dense FP4 tensor-core loop ends without a timeout, its time grows
    in proportion to the MMAs issued, and its rate lies between the BF16
    nominal peak (a dense FP4 rate below it means the loop is not running on
    the FP4 path) and twice NVIDIA's dense FP4 figure for the part."""
    L = _lib.load()
    pairs = int(L.nvfp4_diag_mma_peak_pairs())
    assert 1 <= pairs <= torch.cuda.get_device_properties(0).multi_processor_count // 2
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ms = {}
    for iters in (4096, 4096, 65536):
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record()
        _lib.check(L.nvfp4_diag_mma_peak(iters, _p(st), None, _stream()), "mma loop")
        c1.record()
        torch.cuda.synchronize()
        ms[iters] = c0.elapsed_time(c1)
    assert int(st.item()) == 0
    ratio = ms[65536] / ms[4096]
    assert 8.0 < ratio < 20.0, ms
    tflops = pairs * 65536 * 2 * 256 * 256 * 64 / (ms[65536] * 1e-3) / 1e12
    assert 2250.0 < tflops < 30000.0, tflops


def test_fp4_mma_loop_clock_record():
    """The loop's clock record: the first pair's span in SM cycles grows with
    the MMAs issued, and the SM clock it implies lies between 0.3 and 2.5 GHz
    (the part's highest clock is 2.07 GHz); cycles per MMA are those of a
    dense tensor core (an M=256 N=256 K=64 pair MMA is 8.4 MFLOP)."""
    L = _lib.load()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    clk = torch.zeros(2, 4, dtype=torch.int64, device="cuda")
    for i, iters in enumerate((4096, 65536)):
        _lib.check(L.nvfp4_diag_mma_peak(iters, _p(st), _p(clk[i]), _stream()), "mma loop")
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    c = clk.cpu().numpy()
    ns, cyc = c[:, 1] - c[:, 0], c[:, 3] - c[:, 2]
    assert (ns > 0).all() and (cyc > 0).all(), c
    mhz = 1e3 * cyc / ns
    assert ((mhz > 300) & (mhz < 2500)).all(), mhz
    per_mma = cyc[1] / 65536
    assert 32 < per_mma < 1024, per_mma
    assert 8.0 < cyc[1] / cyc[0] < 20.0, cyc


def _e4m3_values():
    """UE4M3 values of codes 1..126: subnormals m * 2^-9, normals (1 + m/8) * 2^(e-7)."""
    c = np.arange(1, 127)
    e, m = c >> 3, c & 7
    return np.where(e == 0, m * 2.0 ** -9, (1 + m / 8.0) * 2.0 ** (e - 7)).astype(np.float32)


def test_element_codes_match_correctly_rounded_quotient_everywhere():
    """Pass 2's element encoder (a multiply by the reciprocal with one fma
    correction step) gives E2M1(RN(h / sc)) for every BF16 global max A, every
    block-scale code and every BF16 h with |h| <= A, both signs (1.3e11 codes)."""
    L = _lib.load()
    counts = torch.zeros(2, dtype=torch.int64, device="cuda")
    first, last = 1, 0x7F7F
    a = first
    while a <= last:
        n = min(2048, last - a + 1)
        _lib.check(L.nvfp4_diag_quotient_codes(a, n, _p(counts), _stream()), "quotient codes")
        a += n
    torch.cuda.synchronize()
    bad, seen = (int(v) for v in counts.cpu())
    # codes compared: the 2 (A + 1) patterns h with |h| <= A, per (max A,
    # scale) pair whose scale is nonzero
    abits = np.arange(first, last + 1, dtype=np.uint32)
    g = (abits << 16).view(np.float32) / np.float32(2688.0)
    sc = _e4m3_values()[None, :] * g[:, None]
    assert seen == int(((sc > 0).sum(axis=1) * 2 * (abits.astype(np.int64) + 1)).sum())
    assert bad == 0


def test_epilogue_silu_equals_table_for_every_gate():
    """The SwiGLU epilogue of nvfp4_fc1_swiglu reads silu from a 6.5 KB
    shared-memory slice of the table (2^-10 <= |g| < 8), takes g itself for
    g >= 8 and reads the table in global memory otherwise; for all 65,536
    gates it must give the table's (correctly rounded) BF16 silu."""
    L = _lib.load()
    tab = torch.empty(65536, dtype=torch.int16, device="cuda")
    epi = torch.empty(65536, dtype=torch.int16, device="cuda")
    _lib.check(L.nvfp4_diag_silu_all(_p(tab), _stream()), "silu table")
    _lib.check(L.nvfp4_diag_silu_epilogue(_p(epi), _stream()), "silu epilogue")
    torch.cuda.synchronize()
    diff = (tab != epi).nonzero().flatten().cpu().numpy()
    assert diff.size == 0, [hex(int(g)) for g in diff[:8]]
