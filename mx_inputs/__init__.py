"""Seeded synthetic inputs for the MX (block-scaled FP8) matrix product.

This module only *makes inputs*: E4M3 element codes and E8M0 scale bytes,
drawn from a seeded ``torch.Generator`` on the CPU in a fixed, documented
order.  It holds none of the product's arithmetic and is the one module that
both the CUDA path's tests/benchmark and the CPU oracle's tests use.

Layouts produced (row-major, contiguous, uint8):
    A  : M x K          As : M x (K/32)     (one scale per 32 K elements)
    B  : K x N          Bs : N x (K/32)

Block quantizer (per run of 32 consecutive K elements of one row of A, or of
one column of B):
    amax  = max |x| over the block
    scale = clamp(127 + ceil(log2(amax / 448)), 0, 254), 127 when amax == 0
    code  = E4M3 cast (round to nearest even) of clamp(x * 2^(127 - scale), -448, 448)
``ceil(log2(.))`` is taken exactly from the binary exponent (``frexp``), so
the choice does not depend on a host's log2 rounding.  The clamp to +-448
happens before the cast because torch's float8_e4m3fn cast gives NaN rather
than saturating past the largest finite value.

The five standard workloads (names used by the tests and the benchmark):
    square_256       M=N=K=256, N(0,1) quantized, FP32 out, use_acc=0, seed 0
    square_4096      M=N=K=4096, N(0,1) quantized, scale bytes replaced by
                     uniform integers in [123,131], FP32 out
    mlp_up_8192x28672x8192
                     A: N(0,1) with 0.1% of entries x50 before quantization;
                     B: N(0, 0.02); BF16 out; pair-CTA mode
    longk_2048_65536 M=N=2048, K=65536 in 4 chunks of 16384 accumulated into
                     one FP32 C; codes uniform over the 254 finite E4M3 codes,
                     scales uniform integers in [120,134]
    ragged_5000x7000x8192
                     Laplace(0,1) quantized, 5% of scale bytes (each of As, Bs
                     independently) forced to 0 or 254 with probability 1/2
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

E4M3_MAX = 448.0


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def quantize_rows(x: torch.Tensor, chunk_rows: int = 2048):
    """Block-quantize a (R, K) float32 tensor along K in blocks of 32.

    Returns (codes uint8 (R, K), scales uint8 (R, K/32)).  Processed in row
    chunks so that large operands do not need several full-size temporaries.
    """
    R, K = x.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    codes = torch.empty((R, K), dtype=torch.uint8)
    scales = torch.empty((R, K // 32), dtype=torch.uint8)
    for r0 in range(0, R, chunk_rows):
        xb = x[r0:r0 + chunk_rows].to(torch.float32).reshape(-1, K // 32, 32)
        amax = xb.abs().amax(dim=2)
        mant, ex = torch.frexp(amax / E4M3_MAX)          # v = mant * 2^ex, mant in [0.5, 1)
        ceil_log2 = torch.where(mant == 0.5, ex - 1, ex)  # exact ceil(log2(v)) for v > 0
        s = torch.where(amax > 0, 127 + ceil_log2, torch.full_like(ex, 127)).clamp(0, 254)
        mult = torch.pow(2.0, (127 - s).to(torch.float64)).to(torch.float32)
        y = (xb * mult.unsqueeze(2)).clamp(-E4M3_MAX, E4M3_MAX)
        codes[r0:r0 + chunk_rows] = y.reshape(-1, K).to(torch.float8_e4m3fn).view(torch.uint8)
        scales[r0:r0 + chunk_rows] = s.to(torch.uint8)
    return codes, scales


def finite_codes(n: int, g: torch.Generator) -> torch.Tensor:
    """n codes uniform over the 254 non-NaN E4M3 byte codes (0x7F, 0xFF excluded)."""
    r = torch.randint(0, 254, (n,), generator=g, dtype=torch.int32)
    return torch.where(r < 127, r, r + 1).to(torch.uint8)


def integer_codes(shape, lo: int, hi: int, g: torch.Generator) -> torch.Tensor:
    """E4M3 codes of uniform integers in [lo, hi] (|v| <= 16 are exact in E4M3)."""
    v = torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int32).to(torch.float32)
    return v.to(torch.float8_e4m3fn).view(torch.uint8)


@dataclass
class Problem:
    """One GEMM problem: operands plus how it is to be called."""
    name: str
    M: int
    N: int
    K: int
    A: torch.Tensor
    As: torch.Tensor
    B: torch.Tensor
    Bs: torch.Tensor
    out_dtype: str = "f32"          # "f32" or "bf16"
    use_acc: bool = False
    mode: str = "auto"              # "auto", "1cta" or "2cta"
    k_chunks: int = 1               # >1: accumulate over K in this many calls
    meta: dict = field(default_factory=dict)

    def chunk(self, c: int):
        """Operands of call c when the K range is split into k_chunks calls
        (each a contiguous copy, since the C interface takes dense operands)."""
        kc = self.K // self.k_chunks
        k0 = kc * c
        return (self.A[:, k0:k0 + kc].contiguous(), self.As[:, k0 // 32:(k0 + kc) // 32].contiguous(),
                self.B[k0:k0 + kc].contiguous(), self.Bs[:, k0 // 32:(k0 + kc) // 32].contiguous(), kc)


def _quant_B_from_cols(bt: torch.Tensor):
    """bt is (N, K): column j of B.  Returns B codes (K, N) and Bs (N, K/32)."""
    codes_t, bs = quantize_rows(bt)
    return codes_t.t().contiguous(), bs


def square_256(seed: int = 0) -> Problem:
    g = _gen(seed)
    M = N = K = 256
    a = torch.randn((M, K), generator=g)
    bt = torch.randn((N, K), generator=g)
    A, As = quantize_rows(a)
    B, Bs = _quant_B_from_cols(bt)
    return Problem("square_256", M, N, K, A, As, B, Bs, "f32", False)


def square_4096(seed: int = 0, size: int = 4096) -> Problem:
    g = _gen(seed)
    M = N = K = size
    a = torch.randn((M, K), generator=g)
    A, As = quantize_rows(a)
    del a
    bt = torch.randn((N, K), generator=g)
    B, Bs = _quant_B_from_cols(bt)
    del bt
    As = torch.randint(123, 132, As.shape, generator=g, dtype=torch.int32).to(torch.uint8)
    Bs = torch.randint(123, 132, Bs.shape, generator=g, dtype=torch.int32).to(torch.uint8)
    return Problem(f"square_{size}", M, N, K, A, As, B, Bs, "f32", False)


def mlp_up(seed: int = 0, M: int = 8192, N: int = 28672, K: int = 8192) -> Problem:
    g = _gen(seed)
    a = torch.randn((M, K), generator=g)
    out = torch.rand((M, K), generator=g) < 0.001
    a = torch.where(out, a * 50.0, a)
    del out
    A, As = quantize_rows(a)
    del a
    # weights drawn column by column of B (i.e. as an N x K matrix), std 0.02
    Bc, Bsc = [], []
    for n0 in range(0, N, 4096):
        bt = torch.randn((min(4096, N - n0), K), generator=g) * 0.02
        c, s = quantize_rows(bt)
        Bc.append(c)
        Bsc.append(s)
        del bt
    codes_t = torch.cat(Bc)
    B = codes_t.t().contiguous()
    Bs = torch.cat(Bsc)
    return Problem(f"mlp_up_{M}x{N}x{K}", M, N, K, A, As, B, Bs, "bf16", False, mode="2cta")


def longk(seed: int = 0, M: int = 2048, N: int = 2048, K: int = 65536, chunks: int = 4) -> Problem:
    g = _gen(seed)
    A = finite_codes(M * K, g).reshape(M, K)
    B = finite_codes(K * N, g).reshape(K, N)
    As = torch.randint(120, 135, (M, K // 32), generator=g, dtype=torch.int32).to(torch.uint8)
    Bs = torch.randint(120, 135, (N, K // 32), generator=g, dtype=torch.int32).to(torch.uint8)
    return Problem(f"longk_{M}_{K}", M, N, K, A, As, B, Bs, "f32", True, k_chunks=chunks)


def ragged(seed: int = 0, M: int = 5000, N: int = 7000, K: int = 8192) -> Problem:
    g = _gen(seed)
    # Laplace draws through the seeded generator: inverse CDF of a uniform
    u = torch.rand((M, K), generator=g, dtype=torch.float64) - 0.5
    a = (-torch.sign(u) * torch.log1p(-2.0 * u.abs())).to(torch.float32)
    del u
    A, As = quantize_rows(a)
    del a
    u = torch.rand((N, K), generator=g, dtype=torch.float64) - 0.5
    bt = (-torch.sign(u) * torch.log1p(-2.0 * u.abs())).to(torch.float32)
    del u
    B, Bs = _quant_B_from_cols(bt)
    del bt
    for s in (As, Bs):
        hit = torch.rand(s.shape, generator=g) < 0.05
        hi = torch.rand(s.shape, generator=g) < 0.5
        ext = torch.where(hi, torch.full_like(s, 254), torch.zeros_like(s))
        s.copy_(torch.where(hit, ext, s))
    return Problem(f"ragged_{M}x{N}x{K}", M, N, K, A, As, B, Bs, "f32", False)


def random_problem(M: int, N: int, K: int, seed: int = 0, kind: str = "normal",
                   scale_lo: int = 120, scale_hi: int = 134, out_dtype: str = "f32",
                   use_acc: bool = False) -> Problem:
    """Small problems for sweeps.

    kind "normal":  N(0,1) block-quantized, then scale bytes uniform in
                    [scale_lo, scale_hi];
    kind "codes":   element codes uniform over the finite codes;
    kind "int":     small integers in [-8, 8] with every scale 127.
    """
    g = _gen(seed)
    if kind == "normal":
        A, As = quantize_rows(torch.randn((M, K), generator=g))
        B, Bs = _quant_B_from_cols(torch.randn((N, K), generator=g))
        As = torch.randint(scale_lo, scale_hi + 1, As.shape, generator=g, dtype=torch.int32).to(torch.uint8)
        Bs = torch.randint(scale_lo, scale_hi + 1, Bs.shape, generator=g, dtype=torch.int32).to(torch.uint8)
    elif kind == "codes":
        A = finite_codes(M * K, g).reshape(M, K)
        B = finite_codes(K * N, g).reshape(K, N)
        As = torch.randint(scale_lo, scale_hi + 1, (M, K // 32), generator=g, dtype=torch.int32).to(torch.uint8)
        Bs = torch.randint(scale_lo, scale_hi + 1, (N, K // 32), generator=g, dtype=torch.int32).to(torch.uint8)
    elif kind == "int":
        A = integer_codes((M, K), -8, 8, g)
        B = integer_codes((K, N), -8, 8, g)
        As = torch.full((M, K // 32), 127, dtype=torch.uint8)
        Bs = torch.full((N, K // 32), 127, dtype=torch.uint8)
    else:
        raise ValueError(kind)
    return Problem(f"{kind}_{M}x{N}x{K}", M, N, K, A, As, B, Bs, out_dtype, use_acc)


def c_init(M: int, N: int, seed: int, out_dtype: str) -> torch.Tensor:
    """A seeded initial C for use_acc tests: N(0,1) values in the output dtype."""
    g = _gen(seed + 7919)
    c = torch.randn((M, N), generator=g)
    return c.to(torch.bfloat16) if out_dtype == "bf16" else c


def skinny(M: int, seed: int = 0, N: int = 8192, K: int = 8192) -> Problem:
    """Decode-like: a few rows of A against a large B.  N(0,1) entries
    block-quantized (A per row, B per column), scale bytes as quantized,
    FP32 out."""
    g = _gen(seed)
    A, As = quantize_rows(torch.randn((M, K), generator=g))
    bt = torch.randn((N, K), generator=g)
    B, Bs = _quant_B_from_cols(bt)
    del bt
    return Problem(f"skinny_{M}x{N}x{K}", M, N, K, A, As, B, Bs, "f32", False)


# bits of the element codes of each format (one code per byte)
FORMAT_BITS = {"e4m3": 8, "e5m2": 8, "e2m3": 6, "e3m2": 6, "e2m1": 4}


def format_codes(fmt: str, shape, g: torch.Generator) -> torch.Tensor:
    """Uniform random element codes of format fmt, one per byte, without the
    E4M3 NaN codes or the E5M2 infinity/NaN codes (sub-byte codes in the low
    bits, the high bits zero)."""
    nb = FORMAT_BITS[fmt]
    c = torch.randint(0, 1 << nb, shape, generator=g, dtype=torch.int32).to(torch.uint8)
    if fmt == "e4m3":
        c[(c & 0x7F) == 0x7F] = 0x3F
    elif fmt == "e5m2":
        c[(c & 0x7C) == 0x7C] = 0x3C
    return c


def with_formats(p: Problem, a_fmt: str, b_fmt: str, seed: int = 0) -> Problem:
    """The same problem shape and scales with A and B redrawn as random codes
    of the given element formats (an E4M3 operand keeps its codes)."""
    g = _gen(seed + 1)
    A = p.A if a_fmt == "e4m3" else format_codes(a_fmt, tuple(p.A.shape), g)
    B = p.B if b_fmt == "e4m3" else format_codes(b_fmt, tuple(p.B.shape), g)
    q = Problem(f"{p.name}_{a_fmt}x{b_fmt}", p.M, p.N, p.K, A, p.As, B, p.Bs, p.out_dtype,
                p.use_acc, p.mode, p.k_chunks, dict(p.meta))
    q.meta["formats"] = (a_fmt, b_fmt)
    return q


WORKLOADS = {
    "square_256": square_256,
    "square_4096": square_4096,
    "mlp_up_8192x28672x8192": mlp_up,
    "longk_2048_65536": longk,
    "ragged_5000x7000x8192": ragged,
    "skinny_1x8192x8192": lambda seed=0: skinny(1, seed),
    "skinny_16x8192x8192": lambda seed=0: skinny(16, seed),
    "skinny_64x8192x8192": lambda seed=0: skinny(64, seed),
    "skinny_128x8192x8192": lambda seed=0: skinny(128, seed),
}


def pack_scales(S, along_cols: bool = False):
    """Rearrange row-major scales into the packed layout of mxgemm.h
    (MXGEMM_SCALES_PACKED): S is n x K/32 uint8, rows of A (along_cols
    False) or columns of B (along_cols True).  Returns the packed bytes (a
    flat uint8 tensor), padding entries 127.  A layout change only: no value
    is computed."""
    import numpy as np
    s = np.ascontiguousarray(S.cpu().numpy() if hasattr(S, "numpy") else S, dtype=np.uint8)
    n, kbn = s.shape
    steps = -(-kbn // 4)
    if along_cols:
        size = -(-n // 256) * steps * 1024
    else:
        size = -(-n // 128) * steps * 512
    out = np.full(size, 127, dtype=np.uint8)
    r = np.arange(n)[:, None]
    kb = np.arange(kbn)[None, :]
    inner = (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
    if along_cols:
        at = (((r // 256) * steps + kb // 4) * 2 + (r // 128) % 2) * 512 + inner
    else:
        at = ((r // 128) * steps + kb // 4) * 512 + inner
    out[at] = s
    return torch.from_numpy(out)



def pack_elements(codes, nbits: int):
    """Rearrange sub-byte element codes (one per byte, code in the low nbits)
    into the packed form of mxgemm.h (MXGEMM_ELEMS_PACKED): every 16
    consecutive elements of a row become one little-endian 128-bit number,
    element i at bits [nbits*i, nbits*i + nbits), stored in the 16 bytes the
    group occupied (the bytes past 2*nbits are zero).  The rows must hold a
    multiple of 16 elements.  A layout change only: no value is computed."""
    import numpy as np
    c = np.ascontiguousarray(codes.cpu().numpy() if hasattr(codes, "numpy") else codes, dtype=np.uint8)
    rows, n = c.shape
    if n % 16:
        raise ValueError("rows of whole 16-element groups only")
    g = (c.reshape(-1, 16) & ((1 << nbits) - 1)).astype(np.uint8)
    bits = ((g[:, :, None] >> np.arange(nbits, dtype=np.uint8)) & 1).reshape(-1, 16 * nbits)
    packed = np.packbits(bits, axis=1, bitorder="little")  # (groups, 2 * nbits) bytes
    out = np.zeros((g.shape[0], 16), dtype=np.uint8)
    out[:, :packed.shape[1]] = packed
    return torch.from_numpy(out.reshape(rows, n))


def pattern_matrix(R: int, C: int, rows=None, device="cpu", chunk_rows: int = 1024) -> torch.Tensor:
    """A deterministic R x C FP32 matrix, exact in FP32 and BF16 alike, for
    problems too large to generate with a CPU random generator:

        x[r, c] = (((7919 r + 104729 c) mod 255) - 127) / 8 * 2^e,
        e = ((r + floor(c / 32)) mod 16) - 8,

    integers of at most 8 significant bits times a power of two that changes
    from block to block of 32 columns and from row to row (so the blocks'
    scales vary).  Integer arithmetic in int64, then one exact conversion.
    ``rows`` (a list of row indices) returns only those rows, computed the
    same way, so that a sample can be rebuilt on the CPU."""
    pow2 = torch.tensor([2.0 ** e for e in range(-8, 8)], dtype=torch.float32, device=device)
    r_all = torch.arange(R, dtype=torch.int64, device=device) if rows is None else \
        torch.as_tensor(rows, dtype=torch.int64, device=device)
    out = torch.empty((r_all.numel(), C), dtype=torch.float32, device=device)
    c = torch.arange(C, dtype=torch.int64, device=device)[None, :]
    for i in range(0, r_all.numel(), chunk_rows):
        r = r_all[i:i + chunk_rows, None]
        k = (r * 7919 + c * 104729) % 255 - 127
        e = (r + c // 32) % 16
        out[i:i + chunk_rows] = k.to(torch.float32) * 0.125 * pow2[e]
    return out
