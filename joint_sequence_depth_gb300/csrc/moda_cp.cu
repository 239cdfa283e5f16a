// Context-parallel pieces on the CUDA cores: the merge of partial forward states and the
// float32 -> storage-type conversion of accumulated gradients.
//
// A query chunk scored against several key chunks (each a moda_fwd_partial call, one of
// them with the chunk's own depth slots) yields one (O_c, lse_c) per key chunk, each the
// softmax over that chunk's keys alone.  The joint softmax over all of them is the
// online-softmax update of frame "Shared online-softmax states preserve the joint
// operator" applied one chunk at a time, in natural-log form:
//     m = max(lse_a, lse_b),  w_a = e^{lse_a - m},  w_b = e^{lse_b - m}
//     O = (w_a O_a + w_b O_b) / (w_a + w_b),  lse = m + ln(w_a + w_b)
// so the state kept between chunks is (O, lse) with O normalised.  Both kernels are
// HBM-bound elementwise passes: each O row is read and written once in float4s, the grid
// is a multiple of the SM count and strides over the rows.
#include "moda_common.cuh"

namespace moda {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void store4(float* p, float4 x) { *reinterpret_cast<float4*>(p) = x; }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 x) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y), b = __floats2bfloat162_rn(x.z, x.w);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&a);
  u.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// A warp covers 32 / (D/4) rows; lane (sub, cl) holds columns 4 cl .. 4 cl + 3 of row sub.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) merge_kernel(const MergeArgs a) {
  constexpr int LPR = D / 4;     // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, cl = lane % LPR;
  const int64_t n_warps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
  const T* part = static_cast<const T*>(a.o_part);
  T* out = static_cast<T*>(a.o_out);
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5); w * RPW < a.rows;
       w += n_warps) {
    const int64_t row = w * RPW + sub;
    const bool valid = row < a.rows;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    float lse = -INFINITY;
    if (valid) {
      const float4 ob = load4(part + row * D + 4 * cl);
      const float lb = a.lse_part[row];
      if (a.first) {
        o = ob;
        lse = lb;
      } else {
        const float4 oa = load4(a.o_acc + row * D + 4 * cl);
        const float la = a.lse_acc[row];
        const float m = fmaxf(la, lb);
        if (m == -INFINITY) {  // neither state holds any weight yet
          o = oa;
        } else {
          const float wa = exp2f((la - m) * kLog2e), wb = exp2f((lb - m) * kLog2e);
          const float inv = 1.f / (wa + wb);
          o = make_float4((wa * oa.x + wb * ob.x) * inv, (wa * oa.y + wb * ob.y) * inv,
                          (wa * oa.z + wb * ob.z) * inv, (wa * oa.w + wb * ob.w) * inv);
          lse = m + log2f(wa + wb) * kLn2;
        }
      }
    }
    // every lane of a row has read lse_acc before its first lane overwrites it
    __syncwarp();
    if (valid) {
      store4(a.o_acc + row * D + 4 * cl, o);
      if (out != nullptr) store4(out + row * D + 4 * cl, o);
      if (cl == 0) a.lse_acc[row] = lse;
    }
  }
}

// Each thread converts kUnroll float4s per pass, all loads first.
constexpr int kUnroll = 2;

template <typename T>
__global__ void __launch_bounds__(kThreads) convert_kernel(int64_t n, const float* src, T* dst) {
  const int64_t n4 = n / 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i0 < n4; i0 += stride * kUnroll) {
    float4 x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (i0 + u * stride < n4) x[u] = load4(src + 4 * (i0 + u * stride));
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (i0 + u * stride < n4) store4(dst + 4 * (i0 + u * stride), x[u]);
  }
  if (blockIdx.x == 0 && threadIdx.x < n - 4 * n4) {
    const int64_t i = 4 * n4 + threadIdx.x;
    dst[i] = from_f32<T>(src[i]);
  }
}

// One wave of resident CTAs (SM count x CTAs per SM at this kernel's register use), fewer
// when the work is smaller; each thread then strides over the rest.
template <typename K>
unsigned grid_for(K kernel, int64_t work_threads) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0)
    sms = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess || per_sm <= 0) per_sm = 1;
  const int64_t want = (work_threads + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  return static_cast<unsigned>(want < 1 ? 1 : (want < cap ? want : cap));
}

template <typename T, int D>
void merge_launch(const MergeArgs& a, cudaStream_t s) {
  const unsigned grid = grid_for(merge_kernel<T, D>, a.rows * (D / 4));
  merge_kernel<T, D><<<grid, kThreads, 0, s>>>(a);
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, int dtype, cudaStream_t s) {
  if (dtype == 0) {
    if (a.d == 64) merge_launch<float, 64>(a, s);
    else merge_launch<float, 128>(a, s);
  } else {
    if (a.d == 64) merge_launch<__nv_bfloat16, 64>(a, s);
    else merge_launch<__nv_bfloat16, 128>(a, s);
  }
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_convert(int64_t n, const float* src, void* dst, int dtype, cudaStream_t s) {
  const int64_t work = n / 4 > 0 ? (n / 4 + kUnroll - 1) / kUnroll : 1;
  if (dtype == 0) {
    convert_kernel<float><<<grid_for(convert_kernel<float>, work), kThreads, 0, s>>>(n, src, static_cast<float*>(dst));
  } else {
    convert_kernel<__nv_bfloat16><<<grid_for(convert_kernel<__nv_bfloat16>, work), kThreads, 0, s>>>(
        n, src, static_cast<__nv_bfloat16*>(dst));
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moda
