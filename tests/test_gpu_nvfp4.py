"""NVFP4: the two-level quantization kernel (bit-exact codes, scale bytes and
tensor scale against the oracle) and the grouped GEMM on the NVFP4 tensor
cores (against the oracle's product of the dequantized operands)."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_bf16_close, assert_fp32_close, gpu_ops, padded_layout, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    return gpu_ops()


def unpack_codes(packed):
    """[rows, cols/2] bytes -> [rows, cols] E2M1 codes (element 2j in the
    low nibble of byte j)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], 2 * p.shape[1]), dtype=np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out


def nvfp4_atoms_to_rowmajor(atoms, rows, cols):
    """NVFP4 scale layout (include/moe.h) -> [rows, cols/16]."""
    atoms = np.asarray(atoms, dtype=np.uint8).reshape(-1)
    r = np.arange(rows)[:, None]
    b = np.arange(cols // 16)[None, :]
    off = ((b // 16) * (rows // 128) + r // 128) * 2048 + ((b // 4) % 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 \
        + b % 4
    return atoms[off]


def _input(rows, cols, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn((rows, cols), generator=g, device="cuda", dtype=torch.float32)
    # row-dependent magnitudes (2^-8 .. 2^8), a zero block and a negligible block
    x *= torch.exp2(torch.randint(-8, 9, (rows, 1), generator=g, device="cuda").float())
    x[3, 16:32] = 0.0
    x[5, 32:48] *= 1e-12
    return x.bfloat16()


@pytest.mark.parametrize("rows,cols", [(128, 256), (384, 512), (1024, 7168)])
def test_nvfp4_quantize_bit_exact(ops, rows, cols):
    x = _input(rows, cols, rows + cols)
    codes, scales, st = ops.nvfp4_quantize(x)
    torch.cuda.synchronize()
    q, s, st_ref = O.nvfp4_quantize_rows(to_np(x))
    assert np.float32(st.item()) == st_ref
    assert np.array_equal(nvfp4_atoms_to_rowmajor(scales.cpu().numpy(), rows, cols), s)
    got = unpack_codes(codes.cpu().numpy())
    assert np.array_equal(got, q), np.argwhere(got != q)[:5]


def test_nvfp4_quantize_zero_tensor(ops):
    x = torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda")
    codes, scales, st = ops.nvfp4_quantize(x)
    torch.cuda.synchronize()
    assert st.item() == 0.0 and not codes.any() and not scales.any()


def test_nvfp4_quantize_rejects_bad_shapes(ops):
    x = torch.zeros((100, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.MoEError):
        ops.nvfp4_quantize(x)
    assert ops.nvfp4_sf_bytes(128, 200) == -1 and ops.nvfp4_sf_bytes(256, 512) == 256 * 512 // 16


def _operands(ops, sizes, N, K, seed):
    """Grouped A (padded layout), per-group weights B_g [N, K]; both
    quantized on the GPU, and their oracle dequantizations."""
    gofs = padded_layout(sizes)
    M = int(gofs[-1]) + 128                 # a tail of rows outside every group
    G = len(sizes)
    A = _input(M, K, seed)
    W = (_input(G * N, K, seed + 1).float() * 0.05).bfloat16()
    aq, asf, ast = ops.nvfp4_quantize(A)
    bq, bsf, bst = ops.nvfp4_quantize(W)
    torch.cuda.synchronize()
    Ad = O.nvfp4_dequantize_rows(unpack_codes(aq.cpu().numpy()), nvfp4_atoms_to_rowmajor(asf.cpu().numpy(), M, K),
                                 np.float32(ast.item()))
    Wd = O.nvfp4_dequantize_rows(unpack_codes(bq.cpu().numpy()),
                                 nvfp4_atoms_to_rowmajor(bsf.cpu().numpy(), G * N, K), np.float32(bst.item()))
    B = np.transpose(Wd.reshape(G, N, K), (0, 2, 1))          # oracle B_g [K, N]
    gofs_t = torch.from_numpy(gofs.astype(np.int32)).cuda()
    return dict(gofs=gofs, gofs_t=gofs_t, M=M, G=G, aq=aq, asf=asf, ast=ast, bq=bq, bsf=bsf, bst=bst, Ad=Ad, B=B)


@pytest.mark.parametrize("sizes,N,K", [
    ([128, 256, 0, 384], 256, 256),
    ([300, 17, 0, 900, 128], 512, 1024),
    ([700, 1500, 260], 2048, 7168),
])
@pytest.mark.parametrize("mode", ["fwd", "dgrad"])
@pytest.mark.parametrize("kernel", ["auto", "pair"])     # the 1-SM kernel (default) and the CTA-pair instance
def test_nvfp4_grouped_gemm_matches_oracle(ops, sizes, N, K, mode, kernel):
    o = _operands(ops, sizes, N, K, sum(sizes) + N)
    m = ops.MOE_GEMM_FWD if mode == "fwd" else ops.MOE_GEMM_DGRAD
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = torch.full((o["M"], N), 7.0, dtype=torch.bfloat16, device="cuda")
    ops.grouped_gemm_nvfp4(m, o["aq"], o["asf"], o["ast"], o["bq"], o["bsf"], o["bst"], o["gofs_t"], o["G"], o["M"],
                           N, K, ops.MOE_EPI_NONE, d, err, opts=ops.gemm_opts(kernel))
    torch.cuda.synchronize()
    assert err.item() == 0
    R = int(o["gofs"][-1])
    ref = O.grouped_gemm(o["Ad"][:R], o["B"], o["gofs"])
    assert_bf16_close(d[:R], ref, what="nvfp4 D")
    assert torch.all(d[R:] == 7.0)                              # rows outside every group untouched


@pytest.mark.parametrize("kernel", ["auto", "pair"])
def test_nvfp4_grouped_gemm_fp32_out(ops, kernel):
    o = _operands(ops, [256, 128, 512], 256, 512, 77)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = ops.grouped_gemm_nvfp4(ops.MOE_GEMM_FWD, o["aq"], o["asf"], o["ast"], o["bq"], o["bsf"], o["bst"],
                               o["gofs_t"], o["G"], o["M"], 256, 512, ops.MOE_EPI_NONE_F32, err=err,
                               opts=ops.gemm_opts(kernel))
    torch.cuda.synchronize()
    assert err.item() == 0
    R = int(o["gofs"][-1])
    assert_fp32_close(d[:R], O.grouped_gemm(o["Ad"][:R], o["B"], o["gofs"]), what="nvfp4 D fp32")


def test_nvfp4_grouped_gemm_bad_offsets(ops):
    o = _operands(ops, [128, 128], 256, 256, 5)
    bad = torch.tensor([0, 100, 256], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.grouped_gemm_nvfp4(ops.MOE_GEMM_FWD, o["aq"], o["asf"], o["ast"], o["bq"], o["bsf"], o["bst"], bad, 2,
                           o["M"], 256, 256, ops.MOE_EPI_NONE, err=err)
    torch.cuda.synchronize()
    assert err.item() == ops.MOE_ERR_BAD_OFFSETS


def _grouped_rows(sizes, cols, seed, extra=256):
    """Row-permuted bf16 matrix: group g's rows at padded_layout offsets,
    zero padding rows, a buffer of a multiple of 256 rows."""
    gofs = padded_layout(sizes)
    rows = (int(gofs[-1]) + extra + 255) // 256 * 256
    x = _input(rows, cols, seed).float()
    for g, m in enumerate(sizes):
        x[int(gofs[g]) + m:int(gofs[g + 1])] = 0.0
    x[int(gofs[-1]):] = 0.0
    return x.bfloat16(), gofs


@pytest.mark.parametrize("sizes,cols", [([128, 0, 384], 128), ([300, 17, 0, 900, 128], 384), ([700, 1500], 2048)])
def test_nvfp4_quantize_cols_bit_exact(ops, sizes, cols):
    x, gofs = _grouped_rows(sizes, cols, sum(sizes) + cols)
    rows = x.shape[0]
    gofs_t = torch.from_numpy(gofs.astype(np.int32)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, st = ops.nvfp4_quantize_cols(x, gofs_t, len(sizes), err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    R = int(gofs[-1])
    xs = to_np(x)
    # the oracle on the ragged groups (padding rows dropped) lays them out at
    # 16-row offsets; the GPU's 128-row layout holds the same blocks
    starts = gofs[:-1]
    ragged = np.concatenate([xs[int(starts[g]):int(starts[g]) + m] for g, m in enumerate(sizes)])
    roff = np.concatenate([[0], np.cumsum(sizes)])
    q, s, st_ref, padded = O.nvfp4_quantize_cols_grouped(ragged, roff)
    assert np.float32(st.item()) == st_ref
    got_q = unpack_codes(codes.cpu().numpy())                   # [cols, rows]
    got_s = nvfp4_atoms_to_rowmajor(scales.cpu().numpy(), cols, rows)
    for g, m in enumerate(sizes):
        nb = (m + 15) // 16
        lo, plo = int(gofs[g]), int(padded[g])
        assert np.array_equal(got_q[:, lo:lo + 16 * nb], q[:, plo:plo + 16 * nb]), g
        assert np.array_equal(got_s[:, lo // 16:lo // 16 + nb], s[:, plo // 16:plo // 16 + nb]), g
        assert not got_q[:, lo + 16 * nb:int(gofs[g + 1])].any()   # whole padding blocks
    assert not got_q[:, R:].any() and not got_s[:, R // 16:].any()


def test_nvfp4_quantize_cols_bad_offsets(ops):
    x = torch.ones((256, 128), dtype=torch.bfloat16, device="cuda")
    bad = torch.tensor([0, 100, 256], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, st = ops.nvfp4_quantize_cols(x, bad, 2, err=err)
    torch.cuda.synchronize()
    assert err.item() == ops.MOE_ERR_BAD_OFFSETS and not codes.any() and st.item() == 0.0


@pytest.mark.parametrize("sizes,M,N", [([128, 256, 0, 384], 256, 256), ([300, 17, 0, 900, 128], 384, 512),
                                       ([700, 1500, 260], 2048, 512)])
def test_nvfp4_wgrad_matches_oracle(ops, sizes, M, N):
    """dB_g = A_g^T G_g over each group's rows, from the columnwise NVFP4
    codes of both row-permuted operands (groups of odd and even numbers of
    128-row tiles, an empty group)."""
    X, gofs = _grouped_rows(sizes, M, 11 + M)
    Y, _ = _grouped_rows(sizes, N, 12 + N)
    K = X.shape[0]
    G = len(sizes)
    gofs_t = torch.from_numpy(gofs.astype(np.int32)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    aq, asf, ast = ops.nvfp4_quantize_cols(X, gofs_t, G, err=err)
    bq, bsf, bst = ops.nvfp4_quantize_cols(Y, gofs_t, G, err=err)
    d = torch.full((G, M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    ops.grouped_gemm_nvfp4(ops.MOE_GEMM_WGRAD, aq, asf, ast, bq, bsf, bst, gofs_t, G, M, N, K, ops.MOE_EPI_NONE, d, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    Ad = O.nvfp4_dequantize_cols(unpack_codes(aq.cpu().numpy()), nvfp4_atoms_to_rowmajor(asf.cpu().numpy(), M, K),
                                 np.float32(ast.item()))                    # [K, M]
    Bd = O.nvfp4_dequantize_cols(unpack_codes(bq.cpu().numpy()), nvfp4_atoms_to_rowmajor(bsf.cpu().numpy(), N, K),
                                 np.float32(bst.item()))                    # [K, N]
    ref = O.grouped_gemm_wgrad(Ad, Bd, gofs)
    for g in range(G):
        if sizes[g] == 0:
            assert torch.all(d[g] == 0)
        else:
            assert_bf16_close(d[g], ref[g], what=f"nvfp4 dW[{g}]")


def test_nvfp4_wgrad_rejects_fp32_output(ops):
    """The weight gradient is written in bf16 (an empty group's tile is
    zero-filled in bf16): fp32 output is refused on the host."""
    X, gofs = _grouped_rows([128, 0], 128, 3)
    gofs_t = torch.from_numpy(gofs.astype(np.int32)).cuda()
    aq, asf, ast = ops.nvfp4_quantize_cols(X, gofs_t, 2)
    with pytest.raises(ops.MoEError):
        ops.grouped_gemm_nvfp4(ops.MOE_GEMM_WGRAD, aq, asf, ast, aq, asf, ast, gofs_t, 2, 128, 256, X.shape[0],
                               ops.MOE_EPI_NONE_F32)

