"""mxgemm_quantize (MX quantization on the GPU) against the oracle's
quantizer, bit for bit: every code and every scale byte, FP32 and BF16
inputs, blocks along rows and down columns (odd column counts take one
column per thread, even ones two), value ranges from FP32
subnormals to 3e38, exact E4M3 ties and all-zero blocks.  Then the
quantized operands feed the GEMM."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

gu = pytest.importorskip("gpu_util")
mx = pytest.importorskip("block_scaled_gemm_gb300")


@pytest.fixture(scope="module")
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_scaled_gemm_gb300 import _build
    _build.build()
    h = mx.mxgemm_create(0)
    yield h
    mx.mxgemm_destroy(h)


def _values(R, C, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((R, C), generator=g)
    # per-row magnitudes over many decades, so scales span most of [0, 254]
    x = x * torch.exp(torch.randn((R, 1), generator=g) * 20).clamp(max=1e36)
    flat = x.view(-1)
    n = flat.numel()
    k = max(1, n // 16)
    idx = torch.randint(0, n, (k,), generator=g)
    flat[idx] = torch.randint(-3584, 3585, (k,), generator=g) / 8.0    # exact ties at scale 127
    idx = torch.randint(0, n, (k,), generator=g)
    flat[idx] = torch.randn(k, generator=g) * 1e-39                      # FP32 subnormals
    if R >= 2 and C >= 32:
        x[0, :32] = 0.0                                                  # an all-zero block
        x[1, :32] = torch.linspace(-3e38, 3e38, 32, dtype=torch.float64).float()  # near FLT_MAX
    return x


def _gpu_quantize(x, along_cols, dtype):
    R, C = x.shape
    X = x.to(dtype).cuda()
    codes = torch.empty((R, C), dtype=torch.uint8, device="cuda")
    sshape = (C, R // 32) if along_cols else (R, C // 32)
    scales = torch.empty(sshape, dtype=torch.uint8, device="cuda")
    mx.mxgemm_quantize(X, R, C, codes, scales, along_cols=along_cols)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("along_cols,R,C", [(False, 77, 320), (False, 1, 32), (False, 513, 4096),
                                            (True, 96, 77), (True, 32, 1), (True, 4096, 515), (True, 64, 130),
                                            # more blocks than one grid covers: grid-stride
                                            # passes, the last one partly live
                                            (False, 4099, 640), (True, 4096, 2600)])
def test_quantize_bit_exact(built, dtype, along_cols, R, C):
    x = _values(R, C, seed=R * 7 + C)
    xin = x.to(dtype)
    codes, scales = _gpu_quantize(x, along_cols, dtype)
    rc, rs = oracle.quantize_e4m3(xin, along_cols=along_cols)
    assert np.array_equal(scales, rs), f"{int((scales != rs).sum())} scale bytes differ"
    assert np.array_equal(codes, rc), f"{int((codes != rc).sum())} codes differ"


def test_quantized_operands_feed_the_gemm(built):
    h = built
    g = torch.Generator().manual_seed(3)
    M, N, K = 300, 264, 512
    a = torch.randn((M, K), generator=g)
    b = torch.randn((K, N), generator=g) * 0.02
    A = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    As = torch.empty((M, K // 32), dtype=torch.uint8, device="cuda")
    B = torch.empty((K, N), dtype=torch.uint8, device="cuda")
    Bs = torch.empty((N, K // 32), dtype=torch.uint8, device="cuda")
    mx.mxgemm_quantize(a.cuda(), M, K, A, As)
    mx.mxgemm_quantize(b.cuda(), K, N, B, Bs, along_cols=True)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    mx.mxgemm_run(h, M, N, K, A, As, B, Bs, C, 0, mx.OUT_F32)
    torch.cuda.synchronize()
    ra, ras = oracle.quantize_e4m3(a)
    rb, rbs = oracle.quantize_e4m3(b, along_cols=True)
    assert np.array_equal(A.cpu().numpy(), ra) and np.array_equal(Bs.cpu().numpy(), rbs)
    ref, bound = oracle.rows(ra, ras, rb, rbs)
    res = oracle.accept(C.cpu().numpy(), ref, bound, "f32")
    assert res["ok"], res
    # and the quantized product is close to the real one
    exact = (a.double() @ b.double()).numpy()
    assert np.max(np.abs(C.cpu().numpy() - exact)) <= 0.1 * np.max(np.abs(exact))


def test_quantize_rejects_bad_arguments(built):
    x = torch.zeros((4, 64), device="cuda")
    c = torch.empty((4, 64), dtype=torch.uint8, device="cuda")
    s = torch.empty((4, 2), dtype=torch.uint8, device="cuda")
    assert mx.mxgemm_quantize(x, 4, 48, c, s, check=False) == mx.ERR_INVALID_VALUE     # C % 32
    assert mx.mxgemm_quantize(x, 4, 64, c, s, along_cols=True, check=False) == mx.ERR_INVALID_VALUE
    assert mx.mxgemm_quantize(x, 4, 64, c, s, x_dtype=5, check=False) == mx.ERR_INVALID_VALUE
    assert mx.mxgemm_quantize(x, 4, 64, c[:, 1:], s, check=False) == mx.ERR_MISALIGNED
    assert mx.mxgemm_quantize(x, 0, 64, c, s, check=False) == mx.OK


# ------------------------------------------------------- stochastic rounding

def _words(R, C, seed):
    rb = np.random.default_rng(seed).integers(0, 2 ** 32, (R, C), dtype=np.uint64).astype(np.uint32)
    rb.flat[::97] = 0                # rounds away whenever the value is off the grid
    rb.flat[1::89] = 0xFFFFFFFF      # truncates
    return rb


def _gpu_quantize_sr(x, rb, along_cols, dtype):
    R, C = x.shape
    X = x.to(dtype).cuda()
    RB = torch.from_numpy(np.ascontiguousarray(rb).view(np.int32)).cuda()
    codes = torch.empty((R, C), dtype=torch.uint8, device="cuda")
    sshape = (C, R // 32) if along_cols else (R, C // 32)
    scales = torch.empty(sshape, dtype=torch.uint8, device="cuda")
    mx.mxgemm_quantize(X, R, C, codes, scales, along_cols=along_cols, rand_bits=RB)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("along_cols,R,C", [(False, 77, 320), (False, 4099, 640), (True, 96, 77),
                                            (True, 64, 130), (True, 4096, 515)])
def test_quantize_stochastic_bit_exact(built, dtype, along_cols, R, C):
    x = _values(R, C, seed=R * 11 + C)
    xin = x.to(dtype)
    rb = _words(R, C, R + 3 * C)
    codes, scales = _gpu_quantize_sr(x, rb, along_cols, dtype)
    rc, rs = oracle.quantize_e4m3(xin, along_cols=along_cols, rand_bits=rb)
    assert np.array_equal(scales, rs), f"{int((scales != rs).sum())} scale bytes differ"
    assert np.array_equal(codes, rc), f"{int((codes != rc).sum())} codes differ"


@pytest.mark.parametrize("along_cols", [False, True])
def test_quantize_stochastic_thresholds(built, along_cols):
    # a block at scale 127 (its largest magnitude 448) with values whose
    # rounding fractions are known exactly; row 0 gets the last word that
    # still rounds up, row 1 the first that does not
    vals = [(1.0625, 2 ** 31), (0.0009765625, 2 ** 31), (0.00146484375, 3 * 2 ** 30),
            (15.5, 2 ** 31), (440.0, 3 * 2 ** 30), (1.00000011920928955, 4096),
            (0.0166015625, 2 ** 31), (-1.0625, 2 ** 31)]
    x = np.zeros((2, 32), dtype=np.float32)
    rb = np.zeros((2, 32), dtype=np.uint32)
    x[:, 31] = 448.0
    for i, (v, t) in enumerate(vals):
        x[:, i] = v
        rb[0, i] = t - 1
        rb[1, i] = t
    if along_cols:  # 32 rows x 2 columns: the same blocks, down the columns
        x, rb = np.ascontiguousarray(x.T), np.ascontiguousarray(rb.T)
    xt = torch.from_numpy(x)
    codes, scales = _gpu_quantize_sr(xt, rb, along_cols, torch.float32)
    rc, rs = oracle.quantize_e4m3(xt, along_cols=along_cols, rand_bits=rb)
    assert np.array_equal(codes, rc) and np.array_equal(scales, rs)
    up = codes[0] if not along_cols else codes[:, 0]
    down = codes[1] if not along_cols else codes[:, 1]
    dec = np.vectorize(oracle.e4m3)
    assert np.all(np.abs(dec(up[:8])) > np.abs(dec(down[:8])))


def test_quantize_stochastic_rejects_bad_words(built):
    x = torch.zeros((4, 64), device="cuda")
    c = torch.empty((4, 64), dtype=torch.uint8, device="cuda")
    s = torch.empty((4, 2), dtype=torch.uint8, device="cuda")
    rb = torch.zeros((4, 65), dtype=torch.int32, device="cuda")
    lib = mx.library()
    assert lib.mxgemm_quantize_sr(x.data_ptr(), mx.IN_F32, 4, 64, 0, None, c.data_ptr(),
                                  s.data_ptr(), None) == mx.ERR_INVALID_VALUE
    assert lib.mxgemm_quantize_sr(x.data_ptr(), mx.IN_F32, 4, 64, 0, rb[:, 1:].data_ptr(),
                                  c.data_ptr(), s.data_ptr(), None) == mx.ERR_MISALIGNED
