"""Tensor-core operand layouts and TMA swizzle, checked on the GPU against host math.

The attention kernels stage K/V tiles with 128-byte-swizzled TMA boxes and feed
tcgen05.mma from shared memory.  These tests build the shared-memory images on the
host (numpy, written from the layout definitions) and check the MMA result against
an exact matmul (small integers, exact in fp32), and the TMA landing pattern
against the swizzle definition: 16-byte chunk c of row r sits at chunk c ^ (r % 8).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_248_gb300 as m
    m.lib()
    return m


def ksw_image(x: np.ndarray) -> np.ndarray:
    """K-major, 128B-swizzled image of a [R][128] bf16 matrix (uint16 bits):
    two halves of 64 columns, each [R][128 bytes] with chunks XOR-swizzled by row."""
    R = x.shape[0]
    img = np.zeros((2, R, 8, 8), dtype=np.uint16)
    for h in range(2):
        for r in range(R):
            for c in range(8):
                img[h, r, c ^ (r % 8)] = x[r, 64 * h + 8 * c:64 * h + 8 * c + 8]
    return img.reshape(-1)


def mn_plain_image(p: np.ndarray) -> np.ndarray:
    """Unswizzled MN-major image of P [K=128][N=16]: 8x8 core matrices (8 K-rows of
    16 bytes), K-groups 128 bytes apart, N-groups 2048 bytes apart."""
    K, N = p.shape
    img = np.zeros(K * N, dtype=np.uint16)
    for k in range(K):
        for n in range(N):
            byte = (k // 8) * 128 + (k % 8) * 16 + (n // 8) * 2048 + (n % 8) * 2
            img[byte // 2] = p[k, n]
    return img


def bf16_bits(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def run(pkv, M, N, a_mn, b_mn, a_layout, a_lbo, a_sbo, b_layout, b_lbo, b_sbo, a_img, b_img, a_off, b_off):
    params = [M, N, a_mn, b_mn, a_layout, a_lbo, a_sbo, b_layout, b_lbo, b_sbo, a_img.nbytes, b_img.nbytes,
              len(a_off)] + list(a_off) + [0] * (8 - len(a_off)) + list(b_off) + [0] * (8 - len(b_off))
    a_t = torch.from_numpy(a_img.view(np.int16).copy()).cuda()
    b_t = torch.from_numpy(b_img.view(np.int16).copy()).cuda()
    d = torch.full((M, N), float("nan"), device="cuda")
    pkv.pkv_umma_selftest(params, a_t, b_t, d)
    torch.cuda.synchronize()
    assert pkv.pkv_get_last_error() == 0
    return d.cpu().numpy()


def small_ints(shape, seed):
    return np.random.default_rng(seed).integers(-3, 4, size=shape).astype(np.float32)


KSTEP_KMAJOR = [(kk // 4) * 16384 + (kk % 4) * 32 for kk in range(8)]


def test_kmajor_a_kmajor_b_n16(pkv):
    # decode S^T = K Q^T: A = K tile [128 keys][128 d], B = Q [16][128 d]
    K = small_ints((128, 128), 1)
    Q = small_ints((16, 128), 2)
    d = run(pkv, 128, 16, 0, 0, 2, 16, 1024, 2, 16, 1024, ksw_image(bf16_bits(K)), ksw_image(bf16_bits(Q)),
            KSTEP_KMAJOR, [(kk // 4) * 2048 + (kk % 4) * 32 for kk in range(8)])
    np.testing.assert_array_equal(d, K @ Q.T)


def test_kmajor_a_kmajor_b_n128(pkv):
    # prefill S = Q K^T: A = Q [128 rows][128 d], B = K [128 keys][128 d]
    Q = small_ints((128, 128), 3)
    K = small_ints((128, 128), 4)
    d = run(pkv, 128, 128, 0, 0, 2, 16, 1024, 2, 16, 1024, ksw_image(bf16_bits(Q)), ksw_image(bf16_bits(K)),
            KSTEP_KMAJOR, KSTEP_KMAJOR)
    np.testing.assert_array_equal(d, Q @ K.T)


@pytest.mark.parametrize("a_lbo,a_sbo,b_lbo,b_sbo", [(16384, 1024, 128, 2048)])
def test_mnmajor_a_mnmajor_plain_b_n16(pkv, a_lbo, a_sbo, b_lbo, b_sbo):
    # decode O^T = V^T P^T: A = V^T (M = d, K = keys) read from the V tile image,
    # B = P^T (K = keys, N = 16 heads) unswizzled MN-major
    V = small_ints((128, 128), 5)
    P = small_ints((128, 16), 6)
    a_img, b_img = ksw_image(bf16_bits(V)), mn_plain_image(bf16_bits(P))
    expect = V.T @ P
    d = run(pkv, 128, 16, 1, 1, 2, a_lbo, a_sbo, 0, b_lbo, b_sbo, a_img, b_img, [kk * 2048 for kk in range(8)],
            [kk * 256 for kk in range(8)])
    if not np.array_equal(d, expect):
        alts = {}
        for (al, asb, bl, bsb) in [(1024, 16384, 128, 2048), (16384, 1024, 2048, 128), (1024, 16384, 2048, 128)]:
            dd = run(pkv, 128, 16, 1, 1, 2, al, asb, 0, bl, bsb, a_img, b_img, [kk * 2048 for kk in range(8)],
                     [kk * 256 for kk in range(8)])
            alts[(al, asb, bl, bsb)] = bool(np.array_equal(dd, expect))
        pytest.fail(f"MN-major layout mismatch; alternatives matched: {alts}")


def test_kmajor_a_mnmajor_b_n128(pkv):
    # prefill O = P V: A = P [128 rows][128 keys] K-major, B = V (K = keys, N = d) MN-major
    P = small_ints((128, 128), 7)
    V = small_ints((128, 128), 8)
    a_img, b_img = ksw_image(bf16_bits(P)), ksw_image(bf16_bits(V))
    expect = P @ V
    d = run(pkv, 128, 128, 0, 1, 2, 16, 1024, 2, 16384, 1024, a_img, b_img, KSTEP_KMAJOR,
            [kk * 2048 for kk in range(8)])
    if not np.array_equal(d, expect):
        dd = run(pkv, 128, 128, 0, 1, 2, 16, 1024, 2, 1024, 16384, a_img, b_img, KSTEP_KMAJOR,
                 [kk * 2048 for kk in range(8)])
        pytest.fail(f"MN-major B mismatch; swapped LBO/SBO matches: {bool(np.array_equal(dd, expect))}")


def test_tmem_a_mnmajor_b_n128(pkv):
    # prefill O = P V with P read from TMEM: lane r holds row r of P, keys 2c and 2c+1
    # packed low/high in 32-bit column c, i.e. the row-major bf16 bits of P; k step kk
    # reads columns 8 kk .. 8 kk + 7.  B = V as above.
    P = small_ints((128, 128), 9)
    V = small_ints((128, 128), 10)
    a_img, b_img = bf16_bits(P).reshape(-1).copy(), ksw_image(bf16_bits(V))
    d = run(pkv, 128, 128, 0, 1, -1, 0, 0, 2, 16384, 1024, a_img, b_img, [8 * kk for kk in range(8)],
            [kk * 2048 for kk in range(8)])
    np.testing.assert_array_equal(d, P @ V)


@pytest.mark.parametrize("row0", [0, 16, 37])
def test_tma_swizzle_128b(pkv, row0):
    rows = 64
    src = (np.arange(rows * 128, dtype=np.int64) * 7 % 32749).astype(np.int16).reshape(rows, 128)
    src_t = torch.from_numpy(src).cuda().view(torch.bfloat16)
    dump = torch.zeros(2048, dtype=torch.int16, device="cuda")
    pkv.pkv_tma_selftest(src_t, row0, dump)
    torch.cuda.synchronize()
    assert pkv.pkv_get_last_error() == 0
    got = dump.cpu().numpy().reshape(2, 16, 8, 8)
    for h in range(2):
        for r in range(16):
            for c in range(8):
                np.testing.assert_array_equal(got[h, r, c ^ (r % 8)],
                                              src[row0 + r, 64 * h + 8 * c:64 * h + 8 * c + 8])


def test_bounded_wait_times_out_and_the_context_stays_usable(pkv):
    # A wait that nothing completes gives up after its limit (1 s): the kernel reports
    # the timeout through the error word and returns -- no trap, no hang -- and the
    # next call on the same context computes correctly.
    import time

    import oracle
    import workloads as wl
    from helpers import bits, compare

    torch.cuda.synchronize()
    assert pkv.pkv_get_last_error() == 0
    t0 = time.time()
    pkv.pkv_wait_selftest()
    torch.cuda.synchronize()
    took = time.time() - t0
    assert pkv.pkv_get_last_error() == pkv.PKV_ERR_TIMEOUT
    assert 0.5 < took < 30
    w = wl.random_case(5, num_seqs=4, max_ctx=300, max_q=40, group=4, num_kv_heads=2, head_dim=128, dtype="bf16")
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    out = pkv.paged_attention(t["q"], t["k_cache"], t["v_cache"], dev(w.block_tables), dev(w.seq_lens),
                              dev(w.query_start_loc), w.scale, w.max_query_len, w.max_seq_len)
    assert pkv.pkv_get_last_error() == 0
    ref = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w.block_tables,
                           w.seq_lens, w.query_start_loc, w.scale)
    compare(out, ref, "bf16", w.name)
