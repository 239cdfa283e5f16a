// Depth-KV write path for bf16 on sm_103a ("Mixture-of-Depths Attention", frame "Reuse
// attention KV; add a projection for FFN inputs", Sec. 2.2 and Table 3): each layer
// appends its contributions to the depth cache kd, vd [B, Hkv, T, S, d] as slots that the
// later layers' joint softmax reads.
//
//   store:    kd[b,g,t,slot,:] = k[b,g,t,:], vd[...] = v[b,g,t,:]   (the attention KV reused)
//   project:  kd[b,g,t,slot,c] = sum_m x[b,t,m] wk[m, g*d + c]       (the FFN input projected)
//             vd[b,g,t,slot,c] = sum_m x[b,t,m] wv[m, g*d + c]
//
// The store is a strided copy (16-byte vectors).  The projection is a tcgen05 GEMM: one
// CTA per 128 positions x 128 output columns of one batch row, computing K and V together
// as one N = 256 product (the x tile is loaded once for both); x and the wk, wv tiles
// arrive by TMA (128-byte swizzle) through a 2-stage ring (two CTAs per SM), one thread
// issues the MMAs (M = 128, N = 256, K = 16 steps, float32 accumulators in TMEM), and the
// epilogue rounds to bf16 once and writes the tiles straight into the slot with TMA stores
// through a tensor map whose rows step over the S slots of a position (the slot scatter).
//
// All waits are bounded (sm103_ptx.cuh); a timeout records MODA_ERR_TIMEOUT.
#include <cudaTypedefs.h>

#include <algorithm>

#include "moda_common.cuh"
#include "sm103_ptx.cuh"

namespace moda {
namespace {

using namespace sm103;

// ---------------------------------------------------------------------------- store
template <int D>
__global__ void __launch_bounds__(256) moda_depth_store_kernel(const DepthWriteArgs a) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  const int64_t rows = static_cast<int64_t>(a.B) * a.Hkv * a.T;
  const int64_t n = rows * CH;
  const uint4* k = static_cast<const uint4*>(a.k);
  const uint4* v = static_cast<const uint4*>(a.v);
  uint4* kd = static_cast<uint4*>(a.kd);
  uint4* vd = static_cast<uint4*>(a.vd);
  // four vectors of k and four of v in flight per thread before any store
  constexpr int U = 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < n; i0 += U * stride) {
    uint4 rk[U], rv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < n) {
        rk[u] = __ldcs(k + i);
        rv[u] = __ldcs(v + i);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < n) {
        const int64_t dst = (i / CH * a.S + a.slot) * CH + i % CH;
        kd[dst] = rk[u];
        vd[dst] = rv[u];
      }
    }
  }
}

// ---------------------------------------------------------------------------- project
constexpr int PM = 128;  // positions per tile
constexpr int PN = 128;  // output columns per tile (of K and of V each)
constexpr int PK = 64;   // reduction step per stage
constexpr int PSTAGE = 2;
constexpr int P_A_BYTES = PM * PK * 2;      // x tile, K-major
constexpr int P_B_BYTES = 2 * PK * PN * 2;  // wk then wv tile: four [64 x 64] MN-major blocks
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
constexpr int P_OFF_BAR = PSTAGE * P_STAGE_BYTES;  // full[PSTAGE], empty[PSTAGE], done
constexpr int P_SMEM = P_OFF_BAR + (2 * PSTAGE + 1) * 8 + 16;

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src_smem, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(map),
               "r"(src_smem), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

struct ProjParams {
  int B, T, Dm, Hkv, d, n_total;  // n_total = Hkv * d
  int* status;
};

// blockIdx: x = column tile, y = position tile, z = b
__global__ void __launch_bounds__(128, 2)
    moda_depth_project_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmWk,
                              const __grid_constant__ CUtensorMap tmWv, const __grid_constant__ CUtensorMap tmKd,
                              const __grid_constant__ CUtensorMap tmVd, const ProjParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) record_status(p.status, kStatusConfig);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * PN, t0 = blockIdx.y * PM;
  const int b = blockIdx.z;
  const int n_k = (p.Dm + PK - 1) / PK;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + P_OFF_BAR);
  uint64_t* empty = full + PSTAGE;
  uint64_t* done = empty + PSTAGE;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P_OFF_BAR + (2 * PSTAGE + 1) * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P_OFF_BAR + (2 * PSTAGE + 1) * 8 + 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < PSTAGE; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * PN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ loads
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmWk);
    prefetch_tmap(&tmWv);
    int issued = 0;
    for (int ks = 0; ks < n_k; ++ks) {
      const int st = ks % PSTAGE, use = ks / PSTAGE;
      if (use > 0 && !mbar_wait(&empty[st], (use - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      uint8_t* dst = smem + st * P_STAGE_BYTES;
      mbar_arrive_expect_tx(&full[st], P_STAGE_BYTES);
      tma_load_3d(dst, &tmX, &full[st], ks * PK, t0, b);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tma_load_2d(dst + P_A_BYTES + c * (PK * 128), c < 2 ? &tmWk : &tmWv, &full[st], n0 + (c & 1) * 64, ks * PK);
      issued = ks + 1;
    }
    if (!ok) {
      *abort_flag = 1;
      record_status(p.status, kStatusTimeout);
      volatile int never = 0;
      for (int ks = std::max(0, issued - PSTAGE); ks < issued; ++ks)
        mbar_wait(&full[ks % PSTAGE], (ks / PSTAGE) & 1, &never);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t IDESC = idesc_bf16(PM, 2 * PN, true);  // B ([wk | wv]) is MN-major
    for (int ks = 0; ks < n_k; ++ks) {
      const int st = ks % PSTAGE;
      if (!mbar_wait(&full[st], (ks / PSTAGE) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t a_desc = sdesc_sw128(sbase + st * P_STAGE_BYTES, 16, 1024);
      const uint64_t b_desc = sdesc_sw128(sbase + st * P_STAGE_BYTES + P_A_BYTES, PK * 128, 1024);
#pragma unroll
      for (int kk = 0; kk < PK / 16; ++kk)
        mma_bf16_ss(tmem, sdesc_add(a_desc, kk * 32), sdesc_add(b_desc, kk * 16 * 128), IDESC,
                    (ks > 0 || kk > 0) ? 1u : 0u);
      mma_commit(&empty[st]);
    }
    if (!ok) {
      *abort_flag = 1;
      record_status(p.status, kStatusTimeout);
    }
    mma_commit(done);  // also the drain: every MMA issued has completed when this arrives
  }
  __syncwarp();
  // ------------------------------------------------------------ epilogue (all 128 threads)
  volatile int never = 0;
  const bool fin = mbar_wait(done, 0, *abort_flag ? &never : abort_flag);
  tc_fence_after();
  if (!fin && threadIdx.x == 0) record_status(p.status, kStatusTimeout);
  const bool good = __syncthreads_and(fin && !*abort_flag);
  if (good) {
    // thread = row = TMEM lane; stage the bf16 tiles in the freed ring as four 64-column
    // SW128 blocks: K columns n0.., n0+64.., then V columns n0.., n0+64..
    const int r = threadIdx.x;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll 1
    for (int half = 0; half < 4; ++half) {
      uint32_t acc[64];
      tmem_ld64(tmem + lane_base + half * 64, acc);
#pragma unroll
      for (int c16 = 0; c16 < 8; ++c16) {
        const uint4 w = make_uint4(pack_bf16(__uint_as_float(acc[8 * c16]), __uint_as_float(acc[8 * c16 + 1])),
                                   pack_bf16(__uint_as_float(acc[8 * c16 + 2]), __uint_as_float(acc[8 * c16 + 3])),
                                   pack_bf16(__uint_as_float(acc[8 * c16 + 4]), __uint_as_float(acc[8 * c16 + 5])),
                                   pack_bf16(__uint_as_float(acc[8 * c16 + 6]), __uint_as_float(acc[8 * c16 + 7])));
        st_shared_v4(sbase + half * (PM * 128) + sw128_offset(r, c16), w);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      // each 64-column block is 64 columns of one head: head n / d, columns n % d
#pragma unroll
      for (int half = 0; half < 4; ++half) {
        const int n = n0 + (half & 1) * 64;
        if (n < p.n_total)
          tma_store_3d(half < 2 ? &tmKd : &tmVd, sbase + half * (PM * 128), n % p.d, t0, b * p.Hkv + n / p.d);
      }
      bulk_commit();
      bulk_wait_all();  // the stores have read the staging tile and written the slot
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * PN);
  }
}

// ---------------------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 dw_encode_fn() {
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
}

bool dw_encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
               const cuuint32_t* box) {
  auto fn = dw_encode_fn();
  if (fn == nullptr) return false;
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int dw_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 1;
  return std::max(n, 1);
}

}  // namespace

cudaError_t launch_depth_store_sm103(const DepthWriteArgs& a, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(a.B) * a.Hkv * a.T * (a.d / 8);
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>((n + 255) / 256, 4LL * dw_sms()));  // 4 x 256 threads per SM
  if (a.d == 64)
    moda_depth_store_kernel<64><<<grid, 256, 0, s>>>(a);
  else
    moda_depth_store_kernel<128><<<grid, 256, 0, s>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_depth_project_sm103(const DepthWriteArgs& a, cudaStream_t s) {
  const int n_total = a.Hkv * a.d;
  CUtensorMap tx, twk, twv, tkd, tvd;
  {  // x [B, T, Dm] as (Dm, T, B); box 64 x 128 x 1
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.Dm), static_cast<cuuint64_t>(a.T),
                                static_cast<cuuint64_t>(a.B)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.Dm) * 2, static_cast<cuuint64_t>(a.T) * a.Dm * 2};
    const cuuint32_t box[3] = {64, PM, 1};
    if (!dw_encode(&tx, a.x, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {  // w [Dm, Hkv*d] as (Hkv*d, Dm); box 64 x 64
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(n_total), static_cast<cuuint64_t>(a.Dm)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(n_total) * 2};
    const cuuint32_t box[2] = {64, PK};
    if (!dw_encode(&twk, a.wk, 2, dims, strides, box) || !dw_encode(&twv, a.wv, 2, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  {  // slot `slot` of kd/vd [B*Hkv, T, S, d] as (d, T, B*Hkv): rows step over the S slots
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.d), static_cast<cuuint64_t>(a.T),
                                static_cast<cuuint64_t>(a.B) * a.Hkv};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.S) * a.d * 2,
                                   static_cast<cuuint64_t>(a.T) * a.S * a.d * 2};
    const cuuint32_t box[3] = {64, PM, 1};
    const size_t off = static_cast<size_t>(a.slot) * a.d * 2;
    if (!dw_encode(&tkd, static_cast<char*>(a.kd) + off, 3, dims, strides, box) ||
        !dw_encode(&tvd, static_cast<char*>(a.vd) + off, 3, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  ProjParams p;
  p.B = a.B;
  p.T = a.T;
  p.Dm = a.Dm;
  p.Hkv = a.Hkv;
  p.d = a.d;
  p.n_total = n_total;
  p.status = a.status;
  static std::atomic<uint64_t> done{0};
  cudaError_t e = ensure_dynamic_smem(moda_depth_project_kernel, P_SMEM, done);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((n_total + PN - 1) / PN), static_cast<unsigned>((a.T + PM - 1) / PM),
                  static_cast<unsigned>(a.B));
  moda_depth_project_kernel<<<grid, 128, P_SMEM, s>>>(tx, twk, twv, tkd, tvd, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moda
