"""Host-side tests of the C ABI: the library loads without a GPU, exports every
function the header declares, and rejects bad arguments with the documented
status codes before touching any device state (so these run on CPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8w8a8.h")


@pytest.fixture(scope="module")
def L():
    from fp8_w8a8_scaled_gb300 import build as b
    b.build()
    import fp8_w8a8_scaled_gb300 as f
    return f.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = _declared_functions()
    for want in ("fp8_scaled_mm", "rmsnorm_quant_fp8", "quant_fp8_per_token", "quant_fp8_static",
                 "fp8_status_string", "fp8_describe_dispatch", "fp8_get_device_error"):
        assert want in names, names


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    import fp8_w8a8_scaled_gb300 as f
    for code in range(6):
        s = f.status_string(code)
        assert s.startswith("FP8_")
    assert f.status_string(99) == "unknown fp8_status"


P = ctypes.c_void_p
GOOD = P(0x10000)          # 16-byte aligned fake device addresses: validation never dereferences them
GOOD2 = P(0x20000)
GOOD3 = P(0x30000)
SC = P(0x40000)
SC2 = P(0x50000)


def mm(L, A=GOOD, B=GOOD2, sa=SC, sb=SC2, gran=0, od=0, M=4, N=64, K=64, out=GOOD3):
    return L.fp8_scaled_mm(A, B, sa, sb, gran, od, M, N, K, out, None)


def test_scaled_mm_validation(L):
    assert mm(L, M=0) == 0                                     # no-op, nothing launched
    assert mm(L, M=0, A=None, out=None) == 0                   # pointers are not needed for M == 0
    assert mm(L, M=-1) == 1
    assert mm(L, N=0) == 1
    assert mm(L, K=0) == 1
    assert mm(L, M=2 ** 31) == 1
    assert mm(L, gran=5) == 1
    assert mm(L, gran=4, M=0) == 0                             # blockwise is a valid granularity
    assert mm(L, gran=4, K=72) == 2
    assert mm(L, gran=-1) == 1
    assert mm(L, od=1) == 3                                    # only bf16 output
    assert mm(L, A=None) == 1
    assert mm(L, B=None) == 1
    assert mm(L, sa=None) == 1
    assert mm(L, sb=None) == 1
    assert mm(L, out=None) == 1
    assert mm(L, A=P(0x10008)) == 2
    assert mm(L, B=P(0x20001)) == 2
    assert mm(L, out=P(0x30004)) == 2
    assert mm(L, sa=P(0x40002)) == 2
    assert mm(L, K=72) == 2                                    # K % 16
    assert mm(L, N=68) == 2                                    # N % 8


def test_scaled_mm_ex_flags(L):
    args = (GOOD, GOOD2, SC, SC2, 0, 0, 4, 64, 64, GOOD3, None)
    assert L.fp8_scaled_mm_ex(*args[:6], 0, *args[7:], 0) == 0       # M == 0 no-op with flags
    assert L.fp8_scaled_mm_ex(*args, 4) == 1                          # unknown flag bit
    assert L.fp8_scaled_mm_ex(*args, 0x100) == 1
    assert L.fp8_scaled_mm_ex(GOOD, GOOD2, SC, SC2, 0, 0, 4, 64, 72, GOOD3, None, 1) == 2


def test_fused_norm_mm_validation(L):
    f = L.fp8_rmsnorm_quant_scaled_mm
    G4, G5 = P(0x60000), P(0x70000)

    def call(x=GOOD, gamma=GOOD2, sa=SC, B=GOOD3, sb=SC2, gran=1, od=0, M=4, N=64, K=64, a=G4, out=G5, flags=0):
        return f(x, gamma, ctypes.c_float(1e-6), sa, B, sb, gran, od, M, N, K, a, out, None, flags)

    assert call(M=0) == 0
    assert call(M=0, x=None, a=None, out=None) == 0
    assert call(gran=2) == 1            # the activation scale is per tensor
    assert call(gran=3) == 1
    assert call(M=-1) == 1
    assert call(K=65552) == 1
    assert call(flags=4) == 1
    assert call(od=1) == 3
    assert call(x=None) == 1
    assert call(gamma=None) == 1
    assert call(a=None) == 1
    assert call(out=None) == 1
    assert call(a=P(0x60008)) == 2
    assert call(gamma=P(0x20004)) == 2
    assert call(K=72) == 2
    assert call(N=68) == 2


def test_add_rmsnorm_validation(L):
    f = L.fp8_add_rmsnorm_quant
    e = ctypes.c_float(1e-6)
    R = P(0x60000)
    assert f(GOOD, R, GOOD2, e, SC, GOOD3, 0, 64, None) == 0
    assert f(GOOD, None, GOOD2, e, SC, GOOD3, 4, 64, None) == 1
    assert f(GOOD, R, GOOD2, e, SC, GOOD3, 4, 65552, None) == 1
    assert f(GOOD, P(0x60008), GOOD2, e, SC, GOOD3, 4, 64, None) == 2
    assert f(GOOD, R, GOOD2, e, SC, GOOD3, 4, 40, None) == 2


def test_silu_mul_quant_validation(L):
    f = L.fp8_silu_mul_quant_per_token
    assert f(GOOD, GOOD2, SC, 0, 64, None) == 0
    assert f(None, GOOD2, SC, 4, 64, None) == 1
    assert f(GOOD, GOOD2, None, 4, 64, None) == 1
    assert f(GOOD, GOOD2, SC, 4, 131072 + 16, None) == 1
    assert f(GOOD, GOOD2, SC, 4, 0, None) == 1
    assert f(GOOD, GOOD2, SC, 4, 40, None) == 2
    assert f(GOOD, P(0x20008), SC, 4, 64, None) == 2


def test_requant_merge_validation(L):
    f = L.fp8_requant_merge
    I64 = ctypes.c_int64

    def call(ptrs, scales, rows, K=64, out=GOOD3, so=SC):
        n = len(rows)
        pa = (ctypes.c_void_p * n)(*ptrs)
        sa = (ctypes.c_void_p * n)(*scales)
        ra = (I64 * n)(*rows)
        return f(ctypes.cast(pa, P), ctypes.cast(sa, P), ctypes.cast(ra, P), n, K, out, so, None)

    # (only invalid calls here: the fake addresses must never reach a launch)
    assert call([0x10000], [0x40000], [4], K=40) == 2
    assert call([0x10008], [0x40000], [4]) == 2
    assert call([0x10000], [0x40002], [4]) == 2
    assert call([0x10000], [0], [4]) == 1
    assert call([0], [0x40000], [4]) == 1
    assert call([0x10000], [0x40000], [-1]) == 1
    assert call([0x10000] * 17, [0x40000] * 17, [1] * 17) == 1
    assert call([0x10000], [0x40000], [4], out=None) == 1


def test_quantiser_validation(L):
    assert L.quant_fp8_static(GOOD, SC, GOOD2, 0, 64, None) == 0
    assert L.quant_fp8_static(None, SC, GOOD2, 4, 64, None) == 1
    assert L.quant_fp8_static(GOOD, None, GOOD2, 4, 64, None) == 1
    assert L.quant_fp8_static(GOOD, SC, GOOD2, 4, 40, None) == 2
    assert L.quant_fp8_static(P(0x10002), SC, GOOD2, 4, 64, None) == 2
    assert L.quant_fp8_static(GOOD, SC, GOOD2, -3, 64, None) == 1
    assert L.quant_fp8_per_token(GOOD, GOOD2, SC, 0, 64, None) == 0
    assert L.quant_fp8_per_token(GOOD, GOOD2, None, 4, 64, None) == 1
    assert L.quant_fp8_per_token(GOOD, P(0x20008), SC, 4, 64, None) == 2
    assert L.quant_fp8_per_token(GOOD, GOOD2, SC, 4, 0, None) == 1
    assert L.quant_fp8_per_token(GOOD, GOOD2, SC, 4, 2 ** 31, None) == 1
    for fn in (L.fp8_quant_per_token_group, L.fp8_quant_weight_block):
        assert fn(GOOD, GOOD2, SC, 0, 64, None) == 0              # no rows: nothing launched
        assert fn(None, GOOD2, SC, 4, 64, None) == 1
        assert fn(GOOD, None, SC, 4, 64, None) == 1
        assert fn(GOOD, GOOD2, None, 4, 64, None) == 1
        assert fn(GOOD, GOOD2, SC, -1, 64, None) == 1
        assert fn(GOOD, GOOD2, SC, 4, 0, None) == 1
        assert fn(GOOD, GOOD2, SC, 4, 2 ** 31, None) == 1
        assert fn(GOOD, GOOD2, SC, 4, 72, None) == 2             # K % 16
        assert fn(P(0x10008), GOOD2, SC, 4, 64, None) == 2
        assert fn(GOOD, P(0x20004), SC, 4, 64, None) == 2
        assert fn(GOOD, GOOD2, P(0x40002), 4, 64, None) == 2
    assert L.rmsnorm_quant_fp8(GOOD, GOOD2, ctypes.c_float(1e-6), SC, GOOD3, 0, 64, None) == 0
    assert L.rmsnorm_quant_fp8(GOOD, None, ctypes.c_float(1e-6), SC, GOOD3, 4, 64, None) == 1
    assert L.rmsnorm_quant_fp8(GOOD, GOOD2, ctypes.c_float(1e-6), SC, GOOD3, 4, 65536 + 16, None) == 1
    assert L.rmsnorm_quant_fp8(GOOD, P(0x20004), ctypes.c_float(1e-6), SC, GOOD3, 4, 64, None) == 2
    assert L.rmsnorm_quant_fp8(GOOD, GOOD2, ctypes.c_float(1e-6), SC, GOOD3, 4, 24, None) == 2


def test_w8a16_validation(L):
    def w16(x=GOOD, W=GOOD2, sb=SC, gran=1, od=0, M=4, N=64, K=64, out=GOOD3, flags=0):
        return L.fp8_w8a16_mm_ex(x, W, sb, gran, od, M, N, K, out, None, flags)
    assert w16(M=0) == 0 and w16(M=0, x=None, out=None) == 0       # no-op, nothing launched
    assert w16(M=-1) == 1 and w16(N=0) == 1 and w16(K=0) == 1 and w16(M=2 ** 31) == 1
    assert w16(gran=2) == 1 and w16(gran=3) == 1 and w16(gran=4) == 1 and w16(gran=-1) == 1
    assert w16(od=1) == 3
    assert w16(flags=4) == 1
    assert w16(x=None) == 1 and w16(W=None) == 1 and w16(sb=None) == 1 and w16(out=None) == 1
    assert w16(x=P(0x10008)) == 2 and w16(W=P(0x20001)) == 2 and w16(out=P(0x30004)) == 2
    assert w16(sb=P(0x40002)) == 2 and w16(K=72) == 2 and w16(N=68) == 2
    assert L.fp8_w8a16_mm(GOOD, GOOD2, SC, 0, 0, 0, 64, 64, GOOD3, None) == 0
    d = L.fp8_w8a16_describe_dispatch
    assert d(0, 64, 64) == 0 and d(-1, 64, 64) == -1 and d(4, 0, 64) == -1
    # one to four tokens whose binary32 copy fits 96 KB: the GEMV (5)
    assert all(d(M, 10240, 5120) == 5 for M in (1, 2, 3, 4))
    assert d(4, 10240, 5120) == 5 and d(4, 10240, 5136) == 3 and d(1, 5120, 17408) == 5
    assert d(1, 10240, 20480) == 5 and d(1, 10240, 20496) == 3 and d(2, 10240, 17408) == 3
    assert all(d(M, 10240, 5120) == 3 for M in (5, 16, 17, 32))
    assert all(d(M, 10240, 5120) == 4 for M in (33, 64, 2048))
    wd = L.fp8_widen_weight
    assert wd(GOOD, SC, 1, 0, 64, GOOD3, None) == 0
    assert wd(None, SC, 1, 4, 64, GOOD3, None) == 1 and wd(GOOD, None, 1, 4, 64, GOOD3, None) == 1
    assert wd(GOOD, SC, 1, 4, 64, None, None) == 1 and wd(GOOD, SC, 2, 4, 64, GOOD3, None) == 1
    assert wd(GOOD, SC, 1, -1, 64, GOOD3, None) == 1 and wd(GOOD, SC, 1, 4, 0, GOOD3, None) == 1
    assert wd(GOOD, SC, 1, 4, 72, GOOD3, None) == 2 and wd(P(0x10008), SC, 1, 4, 64, GOOD3, None) == 2


def test_selftest_validation(L):
    L.fp8_selftest_bounded_wait.argtypes = [ctypes.c_uint32, ctypes.c_void_p]
    assert L.fp8_selftest_bounded_wait(0, None) == 1
    assert L.fp8_selftest_bounded_wait(3000000, None) == 1


def test_describe_dispatch_is_pure(L):
    assert L.fp8_describe_dispatch(0, 64, 64, 0) == 0
    assert L.fp8_describe_dispatch(-1, 64, 64, 0) == -1
    assert L.fp8_describe_dispatch(4, 64, 64, 7) == -1
    assert L.fp8_describe_dispatch(4, 64, 64, 5) == -1
    assert L.fp8_describe_dispatch(32, 10240, 5120, 4) == 1        # blockwise: same split as the others
    assert L.fp8_describe_dispatch(33, 10240, 5120, 4) == 2
    for M in (1, 2, 4, 8, 16, 17, 24, 32):
        assert L.fp8_describe_dispatch(M, 10240, 5120, 1) == 1
    for M in (33, 64, 65, 128, 2048, 8192):
        assert L.fp8_describe_dispatch(M, 10240, 5120, 1) == 2
        assert L.fp8_describe_dispatch(M, 34816, 5120, 2) == 2
    # the decode kernel's exact sum holds fewer than 2048 k-blocks; longer K
    # goes to the tile kernel (blockwise scaling keeps the decode kernel)
    assert L.fp8_describe_dispatch(1, 8, 2048 * 128, 1) == 2
    assert L.fp8_describe_dispatch(1, 8, 2047 * 128, 1) == 1
    assert L.fp8_describe_dispatch(1, 8, 2048 * 128, 4) == 1
    # the same question twice gives the same answer (no hidden state)
    for M in (1, 33, 127, 128, 129, 2048, 8192):
        assert L.fp8_describe_dispatch(M, 10240, 5120, 2) == L.fp8_describe_dispatch(M, 10240, 5120, 2)


def test_decode_planner(L):
    """Cluster mode (S = floor(floor(8 * SMs / 5) / tiles) CTAs per
    128-channel tile, at least 1, at most the tile's k-blocks, 1 when K has
    at most two k-blocks) when S <= 8; else two persistent CTAs per SM
    (stream-K; never more CTAs than units of one tile x one 128-wide k-block,
    and at most 8 CTAs per tile).  The same plan for every granularity; the
    k-block sums are exact for all but blockwise scaling."""
    f, sp, ex = L.fp8_decode_ctas_for_sms, L.fp8_decode_split_for_sms, L.fp8_decode_exact_for_sms
    for g in (0, 1, 2, 3, 4):
        assert ex(1, 10240, 5120, g, 152) == (0 if g == 4 else 1)
        # cluster mode (243 CTAs' worth of tiles on 152 SMs)
        for M in (1, 16):
            assert sp(M, 10240, 5120, g, 152) == 3 and f(M, 10240, 5120, g, 152) == 80 * 3
        assert sp(16, 34816, 5120, g, 152) == 1 and f(16, 34816, 5120, g, 152) == 272    # whole tiles
        assert sp(8, 5120, 8192, g, 152) == 6 and f(8, 5120, 8192, g, 152) == 40 * 6
        assert sp(8, 5120, 17408, g, 152) == 6
        assert sp(1, 8192, 5120, g, 152) == 3 and sp(1, 7168, 5120, g, 152) == 4 and sp(1, 6144, 5120, g, 152) == 5
        assert sp(1, 4096, 5120, g, 152) == 7 and sp(1, 3840, 5120, g, 152) == 8 and sp(1, 3456, 5120, g, 152) == 0
        assert sp(1, 10240, 384, g, 152) == 3                     # capped at the 3 k-blocks of K
        assert sp(1, 12800, 384, g, 152) == 2
        assert sp(1, 10240, 256, g, 152) == 1 and f(1, 10240, 256, g, 152) == 80   # K of 1-2 k-blocks: whole tiles
        assert sp(4, 512, 256, g, 152) == 1 and f(4, 512, 256, g, 152) == 4
        assert sp(1, 8, 16, g, 152) == 1 and f(1, 8, 16, g, 152) == 1           # one unit
        # stream-K: few tiles with long K ranges
        assert sp(1, 128, 5120, g, 152) == 0
        assert f(1, 128, 5120, g, 152) == 40 // 6                 # at least ceil(40/7) = 6 k-blocks per CTA
        assert sp(1, 8, 65536, g, 152) == 0 and f(1, 8, 65536, g, 152) == 512 // 74
        assert sp(16, 2048, 5120, g, 152) == 0 and f(16, 2048, 5120, g, 152) == 16 * 40 // 6
        assert sp(5, 1032, 5120, g, 152) == 0
        assert sp(32, 10240, 5120, g, 152) == 3 and f(17, 10240, 5120, g, 152) == 240   # the 32-token tile
    assert f(0, 8, 16, 1, 152) == -1 and sp(0, 8, 16, 1, 152) == -1 and sp(33, 10240, 5120, 1, 152) == -1
    assert ex(1, 8, 2048 * 128, 1, 152) == -1                 # 2048 k-blocks: the tile kernel
    assert ex(1, 8, 2047 * 128, 1, 152) == 1
    assert ex(1, 8, 2048 * 128, 4, 152) == 0                  # blockwise has no such limit


def test_decode_planner_properties(L):
    """Random decode shapes, granularities and SM counts: cluster mode takes
    S = the floor rule (at least 1, at most the k-blocks, 1 when K has at
    most two k-blocks) with ceil(N/128) * S CTAs whenever that S is at most
    8; else stream-K with at most two CTAs per SM, never more CTAs than units,
    and at least ceil(kb / 7) units per CTA (so at most 8 CTAs share a tile);
    exact sums for every granularity but blockwise."""
    import random
    rnd = random.Random(5)
    f, sp, ex = L.fp8_decode_ctas_for_sms, L.fp8_decode_split_for_sms, L.fp8_decode_exact_for_sms
    seen = set()
    for _ in range(3000):
        M, N, K = rnd.randint(1, 32), 8 * rnd.randint(1, 8000), 16 * rnd.randint(1, 4096)
        sms = rnd.choice((1, 8, 132, 148, 152, 160))
        g = rnd.choice((0, 1, 2, 3, 4))
        tiles, kb = -(-N // 128), -(-K // 128)
        S, c = sp(M, N, K, g, sms), f(M, N, K, g, sms)
        assert ex(M, N, K, g, sms) == (0 if g == 4 else 1)
        rule = 1 if kb <= 2 else max(1, min((8 * sms // 5) // tiles, kb))
        if rule <= 8:
            assert (S, c) == (rule, tiles * rule), (M, N, K, sms)
        else:
            units = tiles * kb
            assert S == 0 and 1 <= c <= min(2 * sms, units), (M, N, K, sms)
            assert units // c >= -(-kb // 7), (M, N, K, sms)
        seen.add(min(S, 2))
    assert seen == {0, 1, 2}


def test_product_path_is_independent_of_the_oracle():
    """The package never imports the oracle (no CPU fallback exists), and a
    missing library is an error, not a silent alternative: loading the
    binding and the library in a fresh interpreter leaves `oracle` unloaded,
    and with the library file pointed elsewhere lib() raises."""
    import subprocess
    import sys
    from fp8_w8a8_scaled_gb300 import build as b
    b.build()
    pkg = os.path.join(ROOT, "fp8_w8a8_scaled_gb300")
    for name in os.listdir(pkg):
        if name.endswith(".py"):
            text = open(os.path.join(pkg, name)).read()
            assert not re.search(r"^\s*(from|import)\s+oracle\b", text, flags=re.M), name
    code = ("import sys; sys.path.insert(0, %r)\n"
            "import fp8_w8a8_scaled_gb300 as f\n"
            "f.lib()\n"
            "assert 'oracle' not in sys.modules, 'oracle imported by the product path'\n"
            "f._lib = None\n"
            "f.lib_path = lambda: '/nonexistent/libfp8w8a8.so'\n"
            "try:\n"
            "    f.lib()\n"
            "except RuntimeError:\n"
            "    print('raised')\n" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip().endswith("raised"), r.stdout
