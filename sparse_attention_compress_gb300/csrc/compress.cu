// Key / value compression by overlapping mean pooling.
//
// [NOSA-Parts] "NOSA-1B core components", core component 1 (Key compressor): keys are
// cut into windows of `kernel` tokens at step `stride` and each window is averaged;
// [NOSA-Triton] "NOSA-1B source walk-through #3", beyond the kernel: kernel 32,
// stride 16 (neighbouring windows overlap by half).
//
// GB300 design: an HBM stream.  A window of `kernel` = R*stride tokens is the sum of R
// consecutive stride-sized partial sums, so each warp walks a run of windows keeping
// the last R partial sums in registers and reads every key row exactly once (plus one
// partial sum of overlap at the run's edge).  Lanes own 16-byte column chunks of the
// [h_kv*d] row, so every warp load is a fully coalesced row segment, and the `stride`
// row loads of one partial sum are all in flight together.
#include "launch.h"

namespace nsa {

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void add(float* acc, const uint4& u) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      acc[2 * i] += f.x;
      acc[2 * i + 1] += f.y;
    }
  }
  static __device__ __forceinline__ uint4 pack(const float* x) {
    uint4 u;
    u.x = pack_bf16(x[0], x[1]);
    u.y = pack_bf16(x[2], x[3]);
    u.z = pack_bf16(x[4], x[5]);
    u.w = pack_bf16(x[6], x[7]);
    return u;
  }
};
template <>
struct Vec<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void add(float* acc, const uint4& u) {
    acc[0] += __uint_as_float(u.x);
    acc[1] += __uint_as_float(u.y);
    acc[2] += __uint_as_float(u.z);
    acc[3] += __uint_as_float(u.w);
  }
  static __device__ __forceinline__ uint4 pack(const float* x) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                      __float_as_uint(x[3]));
  }
};

constexpr int kMaxWindowsPerWarp = 16;
constexpr int kCompressWarps = 4;

// grid: (ceil(max n_c / (wpw*kCompressWarps)), n_seqs); each warp takes a run of wpw
// windows (wpw <= 16, chosen by the launcher so that the grid fills the GPU).  Stride <= 32.
template <typename T, int R>
__global__ void __launch_bounds__(kCompressWarps * 32, 3) compress_kernel(const T* __restrict__ k, T* __restrict__ kc,
                                                                      Seqs s, int chunks, int stride,
                                                                      float fkernel, int wpw) {
  using V = Vec<T>;
  const int sq = blockIdx.y;
  const int L = seq_len(s, sq);
  const int kernel = R * stride;
  const int n_c = num_cmp(L, kernel, stride);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c_begin = (blockIdx.x * kCompressWarps + warp) * wpw;
  if (c_begin >= n_c) return;
  const int c_end = min(n_c, c_begin + wpw);
  const int64_t start = seq_start(s, sq);
  const int64_t out0 = cmp_offset(s, sq, kernel, stride);
  const uint4* src = reinterpret_cast<const uint4*>(k);
  uint4* dst = reinterpret_cast<uint4*>(kc);

  for (int ch = lane; ch < chunks; ch += 32) {
    float part[R][V::N];  // the R most recent partial sums, part[R-1] newest
#pragma unroll
    for (int a = 0; a < R; ++a)
#pragma unroll
      for (int e = 0; e < V::N; ++e) part[a][e] = 0.f;
    // partial sum u covers tokens u*stride .. u*stride+stride-1; window c = sum of u = c..c+R-1
    for (int u = c_begin; u < c_end + R - 1; ++u) {
#pragma unroll
      for (int a = 0; a + 1 < R; ++a)
#pragma unroll
        for (int e = 0; e < V::N; ++e) part[a][e] = part[a + 1][e];
      float acc[V::N];
#pragma unroll
      for (int e = 0; e < V::N; ++e) acc[e] = 0.f;
      const int64_t row0 = start + (int64_t)u * stride;
      uint4 buf[16];  // the rows of one partial sum are in flight together
      for (int i0 = 0; i0 < stride; i0 += 16) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i0 + i < stride) buf[i] = __ldg(src + (row0 + i0 + i) * chunks + ch);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i0 + i < stride) V::add(acc, buf[i]);
      }
#pragma unroll
      for (int e = 0; e < V::N; ++e) part[R - 1][e] = acc[e];
      const int c = u - (R - 1);
      if (c >= c_begin) {
        float w[V::N];
#pragma unroll
        for (int e = 0; e < V::N; ++e) {
          float x = 0.f;
#pragma unroll
          for (int a = 0; a < R; ++a) x += part[a][e];
          w[e] = x / fkernel;
        }
        dst[(out0 + c) * chunks + ch] = V::pack(w);
      }
    }
  }
}

cudaError_t launch_compress(const Seqs& s, const void* k, void* k_cmp, int hkv, int d, int dtype,
                            int kernel, int stride, cudaStream_t st) {
  const int R = kernel / stride;
  const int n_c_max = s.max_len >= kernel ? (s.max_len - kernel) / stride + 1 : 0;
  if (n_c_max == 0 || s.n_seqs == 0) return cudaSuccess;
  // windows per warp: long runs read each key row once (plus one partial sum of overlap
  // per run), short runs give more warps; take the longest run (<= 16) that still gives
  // about 32 warps per SM for the total number of windows
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t windows = (int64_t)s.n_seqs * n_c_max;  // an upper bound for packed sequences
  int wpw = (int)(windows / ((int64_t)sms * 32));
  wpw = wpw < 1 ? 1 : (wpw > kMaxWindowsPerWarp ? kMaxWindowsPerWarp : wpw);
  const int per_cta = wpw * kCompressWarps;
  dim3 grid((n_c_max + per_cta - 1) / per_cta, s.n_seqs);
  const float inv = (float)kernel;  // the kernel divides the window sum by this
  const int threads = kCompressWarps * 32;
  if (dtype == kBF16) {
    const int chunks = hkv * d / 8;
    using T = __nv_bfloat16;
    switch (R) {
      case 1: compress_kernel<T, 1><<<grid, threads, 0, st>>>((const T*)k, (T*)k_cmp, s, chunks, stride, inv, wpw); break;
      case 2: compress_kernel<T, 2><<<grid, threads, 0, st>>>((const T*)k, (T*)k_cmp, s, chunks, stride, inv, wpw); break;
      case 3: compress_kernel<T, 3><<<grid, threads, 0, st>>>((const T*)k, (T*)k_cmp, s, chunks, stride, inv, wpw); break;
      default: compress_kernel<T, 4><<<grid, threads, 0, st>>>((const T*)k, (T*)k_cmp, s, chunks, stride, inv, wpw); break;
    }
  } else {
    const int chunks = hkv * d / 4;
    using T = float;
    switch (R) {
      case 1: compress_kernel<T, 1><<<grid, threads, 0, st>>>((const T*)k, (T*)k_cmp, s, chunks, stride, inv, wpw); break;
      case 2: compress_kernel<T, 2><<<grid, threads, 0, st>>>((const T*)k, (T*)k_cmp, s, chunks, stride, inv, wpw); break;
      case 3: compress_kernel<T, 3><<<grid, threads, 0, st>>>((const T*)k, (T*)k_cmp, s, chunks, stride, inv, wpw); break;
      default: compress_kernel<T, 4><<<grid, threads, 0, st>>>((const T*)k, (T*)k_cmp, s, chunks, stride, inv, wpw); break;
    }
  }
  return cudaGetLastError();
}

}  // namespace nsa
