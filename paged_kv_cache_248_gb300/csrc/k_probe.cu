// k_probe.cu -- self-tests of the tcgen05 operand layouts and of TMA swizzled loads.
//
// The attention kernels feed tcgen05.mma from shared memory through 64-bit matrix
// descriptors (or, for the A operand, from TMEM) and stage K/V with 128-byte-swizzled
// TMA boxes.  These two small kernels exercise exactly those mechanisms on
// caller-given operand images so the layouts can be checked against a host matmul,
// independent of any attention code.
#include <cstring>

#include "ptx.cuh"
#include "pkv_internal.cuh"

namespace pkv {
namespace {

struct UmmaProbe {
  int32_t M, N, a_mn, b_mn, a_layout, a_lbo, a_sbo, b_layout, b_lbo, b_sbo, a_bytes, b_bytes, k_steps;
  int32_t a_off[8], b_off[8];
};

constexpr int kProbeSmem = 64 * 1024 * 2 + 2048;

__global__ void __launch_bounds__(128) umma_probe_kernel(UmmaProbe P, const uint4* __restrict__ a_img,
                                                         const uint4* __restrict__ b_img, float* __restrict__ d,
                                                         uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* a_s = smem_raw + (base - raw);
  uint8_t* b_s = a_s + 65536;
  for (int i = threadIdx.x; i < P.a_bytes / 16; i += blockDim.x) reinterpret_cast<uint4*>(a_s)[i] = a_img[i];
  for (int i = threadIdx.x; i < P.b_bytes / 16; i += blockDim.x) reinterpret_cast<uint4*>(b_s)[i] = b_img[i];
  fence_proxy_async_smem();
  const int warp = threadIdx.x / 32;
  // a_layout < 0: A comes from TMEM, a_img being [128 rows][acols] 32-bit columns
  // (two bf16 each) that land in columns [N, N + acols) of the rows' lanes
  const bool a_tm = P.a_layout < 0;
  const int acols = a_tm ? P.a_bytes / (128 * 4) : 0;
  uint32_t ncols = 32;
  while (ncols < static_cast<uint32_t>(P.N + acols)) ncols <<= 1;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (a_tm) {
    const uint32_t lane_base = (static_cast<uint32_t>(warp % 4) * 32u) << 16;
    const int row = (warp % 4) * 32 + threadIdx.x % 32;
    const uint32_t* a_rows = reinterpret_cast<const uint32_t*>(a_img);
    for (int c0 = 0; c0 < acols; c0 += 16) {
      uint32_t r[16];
      for (int j = 0; j < 16; ++j) r[j] = a_rows[row * acols + c0 + j];
      tmem_st16(tmem + lane_base + static_cast<uint32_t>(P.N + c0), r);
    }
    tmem_st_wait();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const uint32_t idesc = umma_idesc_bf16(P.M, P.N, P.a_mn != 0, P.b_mn != 0);
    const uint64_t b0 = umma_smem_desc(smem_u32(b_s), P.b_lbo, P.b_sbo, P.b_layout);
    if (a_tm) {
      for (int k = 0; k < P.k_steps; ++k)
        umma_f16_ts(tmem, tmem + static_cast<uint32_t>(P.N + P.a_off[k]), umma_desc_advance(b0, P.b_off[k]), idesc,
                    k > 0);
    } else {
      const uint64_t a0 = umma_smem_desc(smem_u32(a_s), P.a_lbo, P.a_sbo, P.a_layout);
      for (int k = 0; k < P.k_steps; ++k)
        umma_f16_ss(tmem, umma_desc_advance(a0, P.a_off[k]), umma_desc_advance(b0, P.b_off[k]), idesc, k > 0);
    }
    umma_commit(&bar);
  }
  const bool ok = mbar_wait(&bar, 0, &abort_flag);
  if (!ok) flag_error(err, kErrTimeout);
  tc_fence_after();
  if (ok) {
    const int row = (warp % 4) * 32 + threadIdx.x % 32;
    for (int c0 = 0; c0 < P.N; c0 += 16) {
      uint32_t r[16];
      tmem_ld16_sync(tmem + ((static_cast<uint32_t>(warp % 4) * 32u) << 16) + static_cast<uint32_t>(c0), r);
      if (row < P.M)
        for (int j = 0; j < 16; ++j) d[row * P.N + c0 + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
    tmem_relinquish();
  }
}

__global__ void __launch_bounds__(32) tma_probe_kernel(const __grid_constant__ CUtensorMap map, int32_t row0,
                                                       uint4* __restrict__ dump, uint32_t* err) {
  __shared__ __align__(1024) uint8_t buf[4096];
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bar, 4096);
    const uint64_t pol = l2_policy_evict_first();
    tma_load_2d(buf, &map, &bar, 0, row0, pol);
    tma_load_2d(buf + 2048, &map, &bar, 64, row0, pol);
  }
  const bool ok = mbar_wait(&bar, 0, nullptr);
  if (!ok) {
    if (threadIdx.x == 0) flag_error(err, kErrTimeout);
    return;
  }
  for (int i = threadIdx.x; i < 256; i += 32) dump[i] = reinterpret_cast<const uint4*>(buf)[i];
}

// One CTA waits on an mbarrier that nothing arrives on: the bounded wait every kernel
// uses gives up after its limit, and the kernel reports a timeout and returns.
__global__ void __launch_bounds__(32) wait_probe_kernel(uint32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (!mbar_wait(&bar, 0, nullptr) && threadIdx.x == 0) flag_error(err, kErrTimeout);
}

}  // namespace

int run_wait_selftest(uint32_t* err, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(err);
  return cuda_status(cudaGetLastError());
}

int run_umma_selftest(const int32_t* params, const void* a_img, const void* b_img, float* d_out, uint32_t* err,
                      cudaStream_t s) {
  UmmaProbe P;
  static_assert(sizeof(UmmaProbe) == 29 * sizeof(int32_t), "probe params");
  std::memcpy(&P, params, sizeof P);
  if (!(P.M == 128) || P.N < 16 || P.N > 256 || P.N % 16 != 0) return PKV_ERR_INVALID_ARG;
  if (P.a_bytes <= 0 || P.a_bytes > 65536 || P.b_bytes <= 0 || P.b_bytes > 65536) return PKV_ERR_INVALID_ARG;
  if (P.a_bytes % 16 || P.b_bytes % 16 || P.k_steps < 1 || P.k_steps > 8) return PKV_ERR_INVALID_ARG;
  if (P.a_layout < 0) {  // A from TMEM: 128 rows of acols columns, each k step 8 columns in
    const int acols = P.a_bytes / (128 * 4);
    if (P.a_bytes != acols * 128 * 4 || acols % 16 || P.N + acols > 512 || P.a_mn) return PKV_ERR_INVALID_ARG;
    for (int k = 0; k < P.k_steps; ++k)
      if (P.a_off[k] < 0 || P.a_off[k] % 8 || P.a_off[k] + 8 > acols) return PKV_ERR_INVALID_ARG;
  }
  for (int k = 0; k < P.k_steps; ++k)
    if ((P.a_layout >= 0 && (P.a_off[k] < 0 || P.a_off[k] >= P.a_bytes || P.a_off[k] % 16)) || P.b_off[k] < 0 ||
        P.b_off[k] >= P.b_bytes || P.b_off[k] % 16)
      return PKV_ERR_INVALID_ARG;
  cudaError_t e = cudaFuncSetAttribute(umma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
  if (e != cudaSuccess) return cuda_status(e);
  umma_probe_kernel<<<1, 128, kProbeSmem, s>>>(P, static_cast<const uint4*>(a_img),
                                               static_cast<const uint4*>(b_img), d_out, err);
  return cuda_status(cudaGetLastError());
}

int run_tma_selftest(const void* src, int64_t rows, int32_t row0, void* dump, uint32_t* err, cudaStream_t s) {
  if (rows < 16 || row0 < 0 || row0 + 16 > rows) return PKV_ERR_INVALID_ARG;
  CUtensorMap map;
  int st = encode_tensor_map_2d(&map, src, 128, static_cast<uint64_t>(rows), 256, 64, 16);
  if (st != PKV_OK) return st;
  tma_probe_kernel<<<1, 32, 0, s>>>(map, row0, static_cast<uint4*>(dump), err);
  return cuda_status(cudaGetLastError());
}

}  // namespace pkv
