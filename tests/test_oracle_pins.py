"""Pins for the CPU oracle: each test checks the oracle against something other
than itself -- values worked by hand from the format definitions, an
independent library decode, closed forms, exact integer and exact-rational
arithmetic, and identities the definition implies.

Together they are chosen so that a plausible slip anywhere in the oracle (a
wrong bias or sign in a decoder, a dropped subnormal, a scale indexed by the
wrong row/column or block, a transposed operand, a lost term of the sum)
fails at least one of them.
"""
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest
import torch

import mx_inputs as mi
import oracle

GOLDEN = Path(__file__).parent / "golden"


def _golden_values():
    rows = []
    for line in (GOLDEN / "e4m3_e8m0_values.txt").read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        fmt, code, val = line.split()
        rows.append((fmt, int(code, 16), float(val)))
    return rows


@pytest.mark.parametrize("fmt,code,val", _golden_values())
def test_decoder_spot_values(fmt, code, val):
    got = oracle.e4m3(code) if fmt == "e4m3" else oracle.e8m0(code)
    if np.isnan(val):
        assert np.isnan(got)
    else:
        assert got == val
        assert np.signbit(got) == np.signbit(val)


def test_e4m3_all_codes_match_library_decode():
    # torch's float8_e4m3fn is an independent implementation of the same format
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3(c) for c in range(256)])
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(ours))
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(lib[~nan], ours[~nan])
    assert np.array_equal(np.signbit(lib[~nan]), np.signbit(ours[~nan]))
    # 254 finite codes, max 448, smallest positive 2^-9 (subnormal)
    fin = ours[~nan]
    assert fin.max() == 448.0 and fin.min() == -448.0
    assert fin[fin > 0].min() == 2.0 ** -9


def test_e8m0_all_codes_closed_form():
    for s in range(255):
        assert oracle.e8m0(s) == float(Fraction(2) ** (s - 127))
    assert np.isnan(oracle.e8m0(255))


def _tiny_cases():
    cases = []
    for line in (GOLDEN / "tiny_cases.txt").read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        name, K, a, b, exact, f32 = [x.strip() for x in line.split("|")]
        cases.append((name, int(K), a, b, float(exact), float(f32)))
    return cases


def _operand_from_blocks(spec: str, K: int):
    codes = np.zeros(K, dtype=np.uint8)
    scales = np.zeros(K // 32, dtype=np.uint8)
    for kb, blk in enumerate(spec.split(",")):
        code, sc = blk.split(":")
        if "@0" in code:
            codes[kb * 32] = int(code.split("@")[0], 16)
        else:
            codes[kb * 32:(kb + 1) * 32] = int(code, 16)
        scales[kb] = int(sc)
    return codes, scales


@pytest.mark.parametrize("name,K,a,b,exact,f32", _tiny_cases())
def test_hand_computed_tiny_cases(name, K, a, b, exact, f32):
    ac, asc = _operand_from_blocks(a, K)
    bc, bsc = _operand_from_blocks(b, K)
    A = ac.reshape(1, K)
    B = bc.reshape(K, 1)
    ref, bound = oracle.rows(A, asc.reshape(1, -1), B, bsc.reshape(1, -1))
    assert ref[0, 0] == exact
    assert float(oracle.round_f32(ref)[0, 0]) == f32
    # every case here has terms of one sign within each block: bound = sum |terms|
    assert bound[0, 0] >= abs(ref[0, 0])


def _decode_lib(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_all_scales_127_is_plain_fp8_matmul():
    p = mi.random_problem(37, 45, 160, seed=3, kind="codes", scale_lo=127, scale_hi=127)
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs)
    lib = _decode_lib(p.A.numpy()) @ _decode_lib(p.B.numpy())
    # same exact products; only the summation order may differ
    assert np.all(np.abs(ref - lib) <= 1e-13 * bound)


def test_exact_small_integers_equal_int64_matmul():
    p = mi.random_problem(29, 51, 4096, seed=5, kind="int")
    ai = _decode_lib(p.A.numpy()).astype(np.int64)
    bi = _decode_lib(p.B.numpy()).astype(np.int64)
    assert np.array_equal(_decode_lib(p.A.numpy()), ai.astype(np.float64))
    ref, _ = oracle.rows(p.A, p.As, p.B, p.Bs)
    assert np.array_equal(ref, (ai @ bi).astype(np.float64))


def test_brute_force_exact_rationals_tiny():
    # every finite code and extreme scales, summed exactly with Fractions
    g = torch.Generator().manual_seed(11)
    M, N, K = 3, 4, 64
    A = mi.finite_codes(M * K, g).reshape(M, K).numpy()
    B = mi.finite_codes(K * N, g).reshape(K, N).numpy()
    choices = np.array([0, 1, 120, 127, 134, 253, 254], dtype=np.uint8)
    As = choices[torch.randint(0, len(choices), (M, K // 32), generator=g).numpy()]
    Bs = choices[torch.randint(0, len(choices), (N, K // 32), generator=g).numpy()]
    ref, bound = oracle.rows(A, As, B, Bs)
    da, db = _decode_lib(A), _decode_lib(B)
    for i in range(M):
        for j in range(N):
            exact = Fraction(0)
            absum = Fraction(0)
            for k in range(K):
                t = (Fraction(da[i, k]) * Fraction(2) ** (int(As[i, k // 32]) - 127)
                     * Fraction(db[k, j]) * Fraction(2) ** (int(Bs[j, k // 32]) - 127))
                exact += t
                absum += abs(t)
            assert float(absum) == pytest.approx(bound[i, j], rel=1e-15)
            # double accumulation: error at most K * 2^-53 * sum|t|
            assert abs(Fraction(ref[i, j]) - exact) <= Fraction(K, 2 ** 53) * absum


def test_scale_shift_linearity_rows_columns_blocks():
    p = mi.random_problem(16, 24, 128, seed=7, kind="normal", scale_lo=124, scale_hi=130)
    ref, _ = oracle.rows(p.A, p.As, p.B, p.Bs)
    # one row of A_scale shifted by d multiplies that row of C by exactly 2^d
    i, d = 5, 3
    As2 = p.As.clone()
    As2[i] += d
    r2, _ = oracle.rows(p.A, As2, p.B, p.Bs)
    assert np.array_equal(r2[i], ref[i] * 2.0 ** d)
    assert np.array_equal(np.delete(r2, i, 0), np.delete(ref, i, 0))
    # one row of B_scale (= column j of B) shifted by d: column j scales by 2^d
    j, d = 17, -4
    Bs2 = p.Bs.clone()
    Bs2[j] = (Bs2[j].to(torch.int32) + d).to(torch.uint8)
    r3, _ = oracle.rows(p.A, p.As, p.B, Bs2)
    assert np.array_equal(r3[:, j], ref[:, j] * 2.0 ** d)
    assert np.array_equal(np.delete(r3, j, 1), np.delete(ref, j, 1))
    # a single k-block: only that block's contribution scales
    kb, d = 2, 2
    A_blk = p.A.clone()
    keep = torch.zeros_like(A_blk)
    keep[:, kb * 32:(kb + 1) * 32] = A_blk[:, kb * 32:(kb + 1) * 32]
    c_blk, _ = oracle.rows(keep, p.As, p.B, p.Bs)
    As3 = p.As.clone()
    As3[:, kb] += d
    c_blk2, _ = oracle.rows(keep, As3, p.B, p.Bs)
    assert np.array_equal(c_blk2, c_blk * 2.0 ** d)


def test_transpose_symmetry():
    # C^T = (B^T with scales Bs) x (A^T with scales As): roles swapped
    p = mi.random_problem(19, 33, 96, seed=9, kind="codes")
    ref, _ = oracle.rows(p.A, p.As, p.B, p.Bs)
    refT, _ = oracle.rows(p.B.t().contiguous(), p.Bs, p.A.t().contiguous(), p.As)
    assert np.array_equal(refT, ref.T)


def test_k_split_additivity_and_use_acc():
    p = mi.random_problem(12, 20, 256, seed=13, kind="codes")
    full, bfull = oracle.rows(p.A, p.As, p.B, p.Bs)
    half = 128
    a1, a2 = p.A[:, :half].contiguous(), p.A[:, half:].contiguous()
    s1, s2 = p.As[:, :half // 32].contiguous(), p.As[:, half // 32:].contiguous()
    b1, b2 = p.B[:half].contiguous(), p.B[half:].contiguous()
    t1, t2 = p.Bs[:, :half // 32].contiguous(), p.Bs[:, half // 32:].contiguous()
    r1, bd1 = oracle.rows(a1, s1, b1, t1)
    r2, bd2 = oracle.rows(a2, s2, b2, t2, c_in=r1)
    assert np.all(np.abs(r2 - full) <= 1e-14 * bfull)
    # with use_acc the bound counts |C_in| itself, which is at most C_in's own bound
    assert np.all(bd2 <= bfull * (1 + 1e-14))
    r2_alone, bd2_alone = oracle.rows(a2, s2, b2, t2)
    assert np.array_equal(r2, r2_alone + r1)
    assert np.array_equal(bd2, bd2_alone + np.abs(r1))


def test_points_match_rows():
    p = mi.random_problem(40, 50, 192, seed=17, kind="codes")
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs)
    I = np.array([0, 39, 7, 20, 39])
    J = np.array([0, 49, 31, 0, 1])
    r, b = oracle.points(p.A, p.As, p.B, p.Bs, I, J)
    assert np.array_equal(r, ref[I, J]) and np.array_equal(b, bound[I, J])


def test_round_bf16_matches_library_on_binary32_inputs():
    # for inputs exactly representable in binary32, torch's fp32 -> bf16
    # conversion (round to nearest even) is an independent reference
    g = torch.Generator().manual_seed(19)
    x = torch.randn(20000, generator=g, dtype=torch.float32) * torch.pow(
        2.0, torch.randint(-140, 130, (20000,), generator=g).to(torch.float32))
    extra = torch.tensor([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 1.0078125, 3.3895314e38,
                          3.39e38, float("inf"), -float("inf"), 1e-40, -3e-39], dtype=torch.float32)
    x = torch.cat([x, extra])
    lib = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = oracle.round_bf16_bits(x.to(torch.float64).numpy())
    assert np.array_equal(lib, ours)


def test_round_bf16_ties_from_double():
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: nearest even is 1.0
    # 1 + 2^-8 + 2^-40 is above the tie: rounds up (a binary32 first step
    # would have lost the 2^-40 and rounded down)
    assert oracle.round_bf16_bits([1.0 + 2 ** -8])[0] == 0x3F80
    assert oracle.round_bf16_bits([1.0 + 2 ** -8 + 2 ** -40])[0] == 0x3F81
    assert oracle.round_bf16_bits([1.0 + 3 * 2 ** -8])[0] == 0x3F82


def test_accept_flags_a_wrong_element():
    p = mi.random_problem(8, 8, 64, seed=23, kind="normal")
    ref, bound = oracle.rows(p.A, p.As, p.B, p.Bs)
    out = oracle.round_f32(ref)
    assert oracle.accept(out, ref, bound, "f32")["ok"]
    bad = out.copy()
    bad[3, 4] += 1e-3 * bound[3, 4]
    st = oracle.accept(bad, ref, bound, "f32")
    assert not st["ok"] and st["first_bad"] == [3, 4]
    # bf16: 2^-8 relative slack
    bits = oracle.round_bf16_bits(ref)
    assert oracle.accept(bits, ref, bound, "bf16")["ok"]


def test_accept_overflow_class():
    ref = np.array([1e45, 1.0])
    bound = np.array([2e45, 1.0])
    assert oracle.accept(np.array([np.inf, 1.0]), ref, bound, "f32")["ok"]
    assert oracle.accept(np.array([np.nan, 1.0]), ref, bound, "f32")["ok"]
    assert not oracle.accept(np.array([np.inf, np.nan]), ref, bound, "f32")["ok"]


def test_quantizer_recipe_roundtrip():
    # the generator's quantizer must give finite codes with |code value| <= 448
    # and reproduce each block within one E4M3 half-ulp after rescaling
    g = torch.Generator().manual_seed(29)
    x = torch.randn(64, 256, generator=g)
    codes, sc = mi.quantize_rows(x)
    dec = _decode_lib(codes.numpy())
    assert np.isfinite(dec).all() and np.abs(dec).max() <= 448
    scale = 2.0 ** (sc.numpy().astype(np.float64) - 127)
    recon = dec * np.repeat(scale, 32, axis=1)
    rel = np.abs(recon - x.numpy()) / np.repeat(scale, 32, axis=1)
    # E4M3 has 3 mantissa bits: half-ulp of a value v is <= |v| * 2^-4,
    # plus the subnormal quantum 2^-10 for small codes
    assert np.all(rel <= np.abs(dec) * 2 ** -4 + 2 ** -10 + 1e-12)
    # the block maximum lands in [224, 448] (pre-rounding it is in (224, 448]):
    # the scale is the smallest power of two that fits the block
    blkmax = np.abs(dec).reshape(64, 8, 32).max(axis=2)
    assert np.all((blkmax >= 224) & (blkmax <= 448))


# ---------------------------------------------------------------- other MX element formats

def _other_format_values():
    out = []
    for line in (GOLDEN / "mx_other_formats_values.txt").read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        fmt, code, val = line.split()
        out.append((fmt, int(code, 16), float(val)))
    return out


@pytest.mark.parametrize("fmt,code,val", _other_format_values())
def test_other_format_spot_values(fmt, code, val):
    got = oracle.decode(fmt, code)
    if np.isnan(val):
        assert np.isnan(got)
    else:
        assert got == val
        assert np.signbit(got) == np.signbit(val)


def test_e5m2_all_codes_match_library_decode():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e5m2).to(torch.float64).numpy()
    ours = np.array([oracle.decode("e5m2", c) for c in range(256)])
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(lib[~nan], ours[~nan])
    assert np.array_equal(np.signbit(lib[~nan]), np.signbit(ours[~nan]))


@pytest.mark.parametrize("fmt,bits,count,vmax", [("e2m3", 6, 64, 7.5), ("e3m2", 6, 64, 28.0),
                                                  ("e2m1", 4, 16, 6.0)])
def test_subbyte_formats_closed_properties(fmt, bits, count, vmax):
    vals = np.array([oracle.decode(fmt, c) for c in range(count)])
    # finite everywhere, symmetric under the sign bit, monotone in the
    # magnitude code, largest value as the specification states
    assert np.all(np.isfinite(vals))
    half = count // 2
    assert np.array_equal(vals[half:], -vals[:half])
    assert np.all(np.diff(vals[:half]) > 0)
    assert vals.max() == vmax
    # the bits above the code are ignored
    for c in range(count):
        assert oracle.decode(fmt, c | (0xFF << bits) & 0xFF) == vals[c]
    # e4m3 values decoded from the same codes differ: the format is honoured
    assert any(oracle.decode("e4m3", c) != vals[c] for c in range(count))


@pytest.mark.parametrize("fa,fb", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e2m3", "e3m2"),
                                   ("e2m1", "e2m1"), ("e2m1", "e4m3")])
def test_mixed_format_product_brute_force(fa, fb):
    # exact rational sums of the decoded values, independent of the LUTs
    # used inside the oracle
    g = torch.Generator().manual_seed(17)
    M, N, K = 2, 3, 64
    limit = {"e4m3": 256, "e5m2": 256, "e2m3": 64, "e3m2": 64, "e2m1": 16}
    def codes(fmt, n):
        c = torch.randint(0, limit[fmt], (n,), generator=g).numpy().astype(np.uint8)
        if fmt == "e4m3":
            c[(c & 0x7F) == 0x7F] = 0x3F   # no NaN codes
        if fmt == "e5m2":
            c[(c & 0x7C) == 0x7C] = 0x3C   # no inf/NaN codes
        return c
    A = codes(fa, M * K).reshape(M, K)
    B = codes(fb, K * N).reshape(K, N)
    As = torch.randint(120, 135, (M, K // 32), generator=g).numpy().astype(np.uint8)
    Bs = torch.randint(120, 135, (N, K // 32), generator=g).numpy().astype(np.uint8)
    ref, bound = oracle.rows(A, As, B, Bs, a_fmt=fa, b_fmt=fb)
    pts_ref, _ = oracle.points(A, As, B, Bs, np.array([0, 1]), np.array([2, 0]), a_fmt=fa, b_fmt=fb)
    assert pts_ref[0] == ref[0, 2] and pts_ref[1] == ref[1, 0]

    def value(fmt, c):
        # written out again from the definition, with Fractions
        spec = {"e4m3": (4, 3, 7), "e5m2": (5, 2, 15), "e2m3": (2, 3, 1), "e3m2": (3, 2, 3),
                "e2m1": (2, 1, 1)}[fmt]
        eb, mb, bias = spec
        s = (c >> (eb + mb)) & 1
        e = (c >> mb) & ((1 << eb) - 1)
        m = c & ((1 << mb) - 1)
        if e == 0:
            v = Fraction(m, 2 ** mb) * Fraction(2) ** (1 - bias)
        else:
            v = (1 + Fraction(m, 2 ** mb)) * Fraction(2) ** (e - bias)
        return -v if s else v

    for i in range(M):
        for j in range(N):
            exact = sum(value(fa, int(A[i, k])) * Fraction(2) ** (int(As[i, k // 32]) - 127)
                        * value(fb, int(B[k, j])) * Fraction(2) ** (int(Bs[j, k // 32]) - 127)
                        for k in range(K))
            absum = sum(abs(value(fa, int(A[i, k])) * value(fb, int(B[k, j])))
                        * Fraction(2) ** (int(As[i, k // 32]) + int(Bs[j, k // 32]) - 254)
                        for k in range(K))
            assert abs(Fraction(ref[i, j]) - exact) <= Fraction(K, 2 ** 53) * absum
            assert float(absum) == pytest.approx(bound[i, j], rel=1e-15)


# ---------------------------------------------------------------- MX quantizer

def test_e4m3_rne_matches_library_cast():
    # torch's float8_e4m3fn cast rounds to nearest even inside +-448
    g = torch.Generator().manual_seed(23)
    x = torch.cat([
        torch.randn(20000, generator=g) * 100,
        torch.randn(20000, generator=g) * 0.01,          # subnormal range
        (torch.randint(-3584, 3585, (20000,), generator=g) / 8.0),  # many exact ties
        torch.tensor([0.0, -0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -11]),
    ]).clamp(-448, 448).to(torch.float32)
    lib = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_rne(float(v)) for v in x.numpy()], dtype=np.uint8)
    assert np.array_equal(lib, ours)


def _quantizer_cases():
    out = []
    for line in (GOLDEN / "mx_quantizer_scales.txt").read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        a, sc = line.split()
        out.append((float(np.float32(float(a))), int(sc)))
    return out


@pytest.mark.parametrize("amax,scale", _quantizer_cases())
def test_quantizer_scale_hand_cases(amax, scale):
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 5] = -amax
    codes, scales = oracle.quantize_e4m3(x)
    assert scales[0, 0] == scale
    # the largest element lands within E4M3's range, at 448 / 2^k scale
    if amax > 0 and 0 < scale < 254:
        v = abs(oracle.e4m3(codes[0, 5])) * 2.0 ** (scale - 127)
        assert v <= 448 * 2.0 ** (scale - 127)
        assert abs(v - amax) <= amax * 2.0 ** -4 + 2.0 ** (scale - 127 - 9)


def test_quantizer_matches_input_recipe_rows_and_columns():
    # the input generator's recipe uses torch's float8 cast: an independent
    # implementation of the same conversion
    g = torch.Generator().manual_seed(29)
    x = torch.randn((96, 256), generator=g) * torch.exp(torch.randn((96, 1), generator=g) * 4)
    codes, scales = oracle.quantize_e4m3(x)
    rc, rs = mi.quantize_rows(x)
    assert np.array_equal(codes, rc.numpy()) and np.array_equal(scales, rs.numpy())
    # down the columns of a K x N matrix = along the rows of its transpose
    xt = x[:, :64].contiguous()               # K = 96, N = 64
    c2, s2 = oracle.quantize_e4m3(xt, along_cols=True)
    rct, rst = mi.quantize_rows(xt.t().contiguous())
    assert np.array_equal(c2, rct.numpy().T) and np.array_equal(s2, rst.numpy())


def test_quantizer_roundtrip_error_bound():
    # decoded value within half an E4M3 step of the scaled input (or the
    # subnormal step), and every block's largest magnitude in (224, 448]
    g = torch.Generator().manual_seed(31)
    x = (torch.randn((8, 320), generator=g) * 37.0).numpy().astype(np.float32)
    codes, scales = oracle.quantize_e4m3(x)
    for r in range(8):
        for c in range(320):
            s = int(scales[r, c // 32])
            y = float(x[r, c]) * 2.0 ** (127 - s)
            d = oracle.e4m3(codes[r, c])
            step = 2.0 ** -9 if abs(y) < 2.0 ** -6 else 2.0 ** (np.floor(np.log2(abs(y))) - 3)
            assert abs(d - y) <= step / 2 + 1e-300
        for b in range(10):
            amax = np.abs(x[r, 32 * b:32 * b + 32]).max() * 2.0 ** (127 - int(scales[r, b]))
            assert 224.0 < amax <= 448.0


# ------------------------------------------------- stochastic rounding (E4M3)

def _sr_cases():
    out = []
    for line in (GOLDEN / "mx_stochastic_rounding.txt").read_text().splitlines():
        line = line.split("#")[0].strip()
        if not line:
            continue
        y, r, code = line.split()
        out.append((float(y), int(r), int(code, 16)))
    return out


@pytest.mark.parametrize("y,r,code", _sr_cases())
def test_stochastic_rounding_hand_cases(y, r, code):
    assert oracle.e4m3_sr(y, r) == code


def _sr_values(n, seed):
    g = torch.Generator().manual_seed(seed)
    y = torch.cat([torch.randn(n, generator=g) * 100, torch.randn(n, generator=g) * 0.01,
                   torch.randn(n, generator=g) * 1e-30,
                   torch.randint(-3584, 3585, (n,), generator=g) / 8.0])
    return y.clamp(-448, 448).to(torch.float32)


def test_stochastic_rounding_brackets_and_matches_nearest():
    # r = 0 rounds away from zero, the largest r toward zero (no value here has
    # a fraction above 1 - 2^-32); the two are the same or adjacent grid
    # points around y, and the library's round-to-nearest lands on one of them
    y = _sr_values(3000, 41)
    rn = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, near in zip(y.numpy(), rn):
        v = float(v)
        up = oracle.e4m3(oracle.e4m3_sr(v, 0))
        down = oracle.e4m3(oracle.e4m3_sr(v, 0xFFFFFFFF))
        a = abs(v)
        q = 2.0 ** -9 if a < 2.0 ** -6 else 2.0 ** (np.floor(np.log2(a)) - 3)
        assert abs(down) <= a <= abs(up)
        assert abs(up) - abs(down) in (0.0, q)
        if abs(up) == abs(down):
            assert abs(up) == a  # only values on the grid are left alone
        assert oracle.e4m3(int(near)) in (up, down) or (a == 0.0)


def test_stochastic_rounding_is_unbiased():
    # over r spread evenly across [0, 2^32), the mean result is y, to within
    # the spread's resolution (q / 4096 for 4096 words)
    rs = [k * (1 << 20) + 777 for k in range(4096)]
    for v in list(_sr_values(8, 47).numpy()) + [1.0625, -0.00146484375, 447.0, 300.1]:
        v = float(v)
        if v == 0.0:
            continue
        a = abs(v)
        q = 2.0 ** -9 if a < 2.0 ** -6 else 2.0 ** (np.floor(np.log2(a)) - 3)
        mean = np.mean([oracle.e4m3(oracle.e4m3_sr(v, r)) for r in rs])
        assert abs(mean - v) <= q / 4096 * 1.0001, (v, mean)


def test_stochastic_quantizer_keeps_scales_and_brackets_codes():
    g = torch.Generator().manual_seed(53)
    x = torch.randn((64, 128), generator=g) * torch.exp(torch.randn((64, 1), generator=g) * 6)
    rb = np.random.default_rng(59).integers(0, 2 ** 32, (64, 128), dtype=np.uint64).astype(np.uint32)
    rn_codes, rn_scales = oracle.quantize_e4m3(x)
    sr_codes, sr_scales = oracle.quantize_e4m3(x, rand_bits=rb)
    up, _ = oracle.quantize_e4m3(x, rand_bits=np.zeros((64, 128), np.uint32))
    down, _ = oracle.quantize_e4m3(x, rand_bits=np.full((64, 128), 0xFFFFFFFF, np.uint32))
    assert np.array_equal(sr_scales, rn_scales)     # the block scale does not depend on r
    dec = np.vectorize(oracle.e4m3)
    for codes in (sr_codes, rn_codes):
        d = np.abs(dec(codes))
        assert np.all((d == np.abs(dec(up))) | (d == np.abs(dec(down))))
    # down the columns = along the rows of the transpose, with the words transposed
    xt = x[:, :64].contiguous()
    c2, s2 = oracle.quantize_e4m3(xt, along_cols=True, rand_bits=rb[:, :64])
    ct, st = oracle.quantize_e4m3(xt.t().contiguous(), rand_bits=np.ascontiguousarray(rb[:, :64].T))
    assert np.array_equal(c2, ct.T) and np.array_equal(s2, st)



def test_stochastic_rounding_against_exact_rationals():
    # the definition again, in exact rationals (no floating point): the E4M3
    # magnitude below |y| on the grid, the fraction of the step above it, and
    # the comparison of r with 2^32 times that fraction; codes come from the
    # decoder's table of the 127 finite magnitudes
    from fractions import Fraction
    table = {Fraction(oracle.e4m3(c)): c for c in range(0x7F)}
    rng = np.random.default_rng(67)
    ys = np.concatenate([rng.standard_normal(300) * 100, rng.standard_normal(300) * 0.01,
                         rng.standard_normal(100) * 1e-35,
                         rng.integers(-3584, 3585, 200) / 8.0]).astype(np.float32)
    rs = rng.integers(0, 2 ** 32, ys.size, dtype=np.uint64)
    rs[::5] = 0
    rs[1::7] = 2 ** 32 - 1
    for yv, r in zip(ys, rs):
        y = Fraction(float(yv))
        a = min(abs(y), Fraction(448))
        sign = 0x80 if float(yv) < 0 or (float(yv) == 0 and np.signbit(yv)) else 0
        if a == 0:
            want = sign
        else:
            e = a.numerator.bit_length() - a.denominator.bit_length()
            if Fraction(2) ** e > a:
                e -= 1                      # now 2^e <= a < 2^(e+1)
            q = Fraction(2) ** (max(e, -6) - 3)
            n = a // q
            frac = a / q - n
            mag = (n + 1) * q if int(r) < frac * 2 ** 32 else n * q
            want = sign | table[mag]
        assert oracle.e4m3_sr(float(yv), int(r)) == want, (float(yv), int(r))


def test_nan_codes_and_scale_255_poison_exactly_their_rows_and_columns():
    # E4M3 codes 0x7F / 0xFF and the E8M0 byte 255 are NaN (reading 2 of the
    # readings; OCP MX v1.0): a NaN element or scale of A poisons its row of
    # C, one of B its column, and nothing else changes
    p = mi.random_problem(40, 48, 128, seed=5, kind="int")
    ref0, _ = oracle.rows(p.A, p.As, p.B, p.Bs)
    A, As, B, Bs = p.A.clone(), p.As.clone(), p.B.clone(), p.Bs.clone()
    A[5, 17] = 0x7F
    A[9, 100] = 0xFF
    As[12, 2] = 255
    B[33, 20] = 0x7F
    Bs[30, 1] = 255
    ref, _ = oracle.rows(A, As, B, Bs)
    mask = np.zeros((40, 48), dtype=bool)
    mask[[5, 9, 12], :] = True
    mask[:, [20, 30]] = True
    assert np.array_equal(np.isnan(ref), mask)
    assert np.array_equal(ref[~mask], ref0[~mask])
