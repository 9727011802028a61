"""GPU parity of nvfp4_quantize_pack against the oracle's quantiser: codes and
atom-layout scales must be bit-identical (integer outputs), for bf16 and fp16
inputs, ragged rows and K tails, the rounding tie points, zero, tiny and
saturating blocks; then quantised activations feed the GEMM."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from nvfp4_block_scaled_grouped_gb300 import build
    build.build_library()
    import nvfp4_block_scaled_grouped_gb300 as nv
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.init()
    return nv


def _host_f32(xt):
    """Exact fp32 values of a bf16 / fp16 CUDA tensor."""
    return xt.float().cpu().numpy()


def _check(nv, oracle_mod, xt, what, rows_sample=None):
    codes, sf = nv.quantize_pack_tensor(xt)
    torch.cuda.synchronize()
    x = _host_f32(xt)
    rows, k = x.shape
    got_codes = codes.cpu().numpy()
    got_sf = sf.cpu().numpy()
    if rows_sample is None:
        ref_codes, ref_sf = oracle_mod.quantize(x)
        np.testing.assert_array_equal(got_codes, ref_codes, err_msg=f"{what}: codes")
        np.testing.assert_array_equal(got_sf, oracle_mod.pack_scales(ref_sf, k), err_msg=f"{what}: scales")
        return got_codes, got_sf
    ref_codes, ref_sf = oracle_mod.quantize(x[rows_sample])
    np.testing.assert_array_equal(got_codes[rows_sample], ref_codes, err_msg=f"{what}: codes")
    for i, r in enumerate(rows_sample):
        for kb in range(k // 16):
            assert got_sf[oracle_mod.scale_atom_offset(int(r), kb, k)] == ref_sf[i, kb], (what, r, kb)
    return got_codes, got_sf


SHAPES = [(1, 16), (5, 48), (128, 64), (130, 96), (257, 80), (64, 1024), (33, 7168)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("rows,k", SHAPES)
def test_random_inputs_bit_exact(nv, oracle_mod, dtype, rows, k):
    g = torch.Generator().manual_seed(1000 * rows + k)
    x = (torch.randn(rows, k, generator=g) * 3).to(dtype).cuda()
    _check(nv, oracle_mod, x, f"{dtype} {rows}x{k}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
def test_tie_points_and_special_blocks(nv, oracle_mod, dtype):
    """Blocks whose elements sit exactly on the e2m1 rounding boundaries for
    several scales, amax values on e4m3 ties, zero / tiny / huge blocks, signed
    zeros."""
    rows, k = 40, 256
    x = np.zeros((rows, k), np.float32)
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    decs = [1.0, 0.5, 1.125, 0.1875, 2.0 ** -7, 0.0390625, 24.0]        # e4m3-representable scales
    for r, dec in enumerate(decs):
        for b in range(k // 16):
            blk = np.zeros(16, np.float32)
            blk[0] = 6.0 * dec                                          # amax / 6 == dec exactly
            vals = np.concatenate([ties, -ties, [0.0]])[: 15]
            blk[1:] = vals * dec * (1 if b % 2 == 0 else -1)
            x[r, 16 * b: 16 * b + 16] = blk
    x[10, :] = 0.0                                                      # all-zero row
    x[11, :] = -1e-7                                                    # scale rounds to 0: +0 codes
    x[12, :16] = 3.1875                                                 # amax/6 = 0.53125, an e4m3 tie
    x[12, 16:32] = 7.125                                                # amax/6 = 1.1875, an e4m3 tie
    x[13, :] = 60000.0 if dtype == torch.float16 else 1e30              # saturating scale
    x[13, ::3] = -x[13, ::3]
    x[14, :] = -0.0
    x[15:, :] = np.random.default_rng(4).normal(0, 1, (rows - 15, k)) * np.logspace(-6, 3.5, rows - 15)[:, None]
    xt = torch.from_numpy(x).to(dtype)
    assert np.array_equal(xt.float().numpy()[:8], x[:8]), "tie values must be exact in the input type"
    _check(nv, oracle_mod, xt.cuda(), f"{dtype} ties")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
def test_every_input_value_under_every_scale(nv, oracle_mod, dtype):
    """Exhaustive over the input type: for each of the 126 non-zero finite e4m3
    scales dec, blocks whose first element is 6 * dec (so the block scale is
    dec) carry every finite value x of the type with |x| <= 9 * dec, both
    signs, in the other 15 places; every code must match the oracle's."""
    if dtype == torch.bfloat16:
        allv = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    else:
        allv = np.arange(1 << 16, dtype=np.uint16).view(np.float16).astype(np.float32)
    allv = np.unique(np.abs(allv[np.isfinite(allv)]))
    blocks = []
    for c in range(1, 0x7F):
        dec = oracle_mod.e4m3fn_value(c)
        if 6.0 * dec > float(torch.finfo(dtype).max):
            continue
        vals = allv[allv <= 9.0 * dec]
        vals = np.concatenate([vals, -vals])
        pad = (-len(vals)) % 15
        vals = np.concatenate([vals, np.zeros(pad, np.float32)]).reshape(-1, 15)
        head = np.full((vals.shape[0], 1), 6.0 * dec, np.float32)
        blocks.append(np.concatenate([head, vals], axis=1))
    x = np.concatenate(blocks).reshape(-1)
    k = 1024
    x = np.concatenate([x, np.zeros((-len(x)) % k, np.float32)]).reshape(-1, k)
    xt = torch.from_numpy(x).to(dtype)
    assert np.array_equal(xt.float().numpy(), x)
    _check(nv, oracle_mod, xt.cuda(), f"exhaustive {dtype}")


def test_padding_bytes_are_zero(nv, oracle_mod):
    rows, k = 70, 80                                                     # 58 padding rows, 3 padding blocks
    x = torch.randn(rows, k, dtype=torch.float32).to(torch.bfloat16).cuda()
    sf = torch.full((nv.scale_bytes(rows, k),), 0xAB, dtype=torch.uint8, device="cuda")
    codes = torch.full((rows, k // 2), 0xCD, dtype=torch.uint8, device="cuda")
    nv.quantize_pack(x.data_ptr(), nv.DTYPE_BF16, rows, k, codes.data_ptr(), sf.data_ptr())
    torch.cuda.synchronize()
    ref_codes, ref_sf = oracle_mod.quantize(x.float().cpu().numpy())
    np.testing.assert_array_equal(codes.cpu().numpy(), ref_codes)
    np.testing.assert_array_equal(sf.cpu().numpy(), oracle_mod.pack_scales(ref_sf, k))   # padding 0x00


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_full_size_activations_sampled(nv, oracle_mod, name):
    """The activation shapes of the decode and prefill workloads (all rows of
    all groups stacked), checked on sampled rows."""
    from nvfp4_block_scaled_grouped_gb300 import workloads
    rows = int(sum(s[0] for s in workloads.problem_sizes(name)))
    k = 7168
    g = torch.Generator().manual_seed(rows)
    x = torch.randn(rows, k, generator=g).to(torch.bfloat16).cuda()
    rng = np.random.default_rng(rows)
    sample = np.unique(np.concatenate([rng.integers(0, rows, 64), [0, rows - 1]]))
    _check(nv, oracle_mod, x, name, rows_sample=sample)


def test_quantised_activations_feed_the_gemm(nv, oracle_mod):
    """Quantise A and B on the GPU, multiply them with the grouped GEMM, and
    compare with the oracle GEMM of the oracle's quantisation of the same
    inputs (identical operand bytes, so the GEMM parity rule applies)."""
    from parity import assert_parity
    m, n, k = 150, 256, 512
    gen = torch.Generator().manual_seed(77)
    xa = torch.randn(m, k, generator=gen).to(torch.bfloat16).cuda()
    xb = torch.randn(n, k, generator=gen).to(torch.float16).cuda()
    a, sfa = nv.quantize_pack_tensor(xa)
    b, sfb = nv.quantize_pack_tensor(xb)
    c = torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda")
    nv.grouped_gemm_tensors([(m, n, k, 1)], [a], [b], [sfa], [sfb], [c])
    torch.cuda.synchronize()
    ra, rsa = oracle_mod.quantize(xa.float().cpu().numpy())
    rb, rsb = oracle_mod.quantize(xb.float().cpu().numpy())
    ref = oracle_mod.grouped_gemm([(m, n, k, 1)], [ra], [rb], [rsa], [rsb])[0]
    assert_parity(c.cpu().numpy(), ref, "quantised GEMM")


def test_quantize_host_argument_errors(nv):
    st = {v: s for s, v in nv.STATUS.items()}
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(4, 32, dtype=torch.uint8, device="cuda")
    s = torch.zeros(512, dtype=torch.uint8, device="cuda")
    q = lambda *a: nv.quantize_pack(*a, check=False)
    assert q(x.data_ptr(), 0, 0, 64, c.data_ptr(), s.data_ptr()) == 0
    assert q(x.data_ptr(), 2, 4, 64, c.data_ptr(), s.data_ptr()) == st["NVFP4_ERR_INVALID_ARG"]
    assert q(x.data_ptr(), 0, 4, 40, c.data_ptr(), s.data_ptr()) == st["NVFP4_ERR_UNSUPPORTED"]
    assert q(x.data_ptr() + 2, 0, 4, 64, c.data_ptr(), s.data_ptr()) == st["NVFP4_ERR_MISALIGNED"]
    assert q(0, 0, 4, 64, c.data_ptr(), s.data_ptr()) == st["NVFP4_ERR_INVALID_ARG"]
