// Micro-benchmarks of the ceilings that bound the hot path on this GPU, printed as one
// JSON object: L2-resident read bandwidth (the gather of selected K/V blocks is served
// from L2), the L2 -> shared-memory gather rate of random 4 KB slices by cp.async (the
// selected-attention access pattern, with no compute), HBM read bandwidth, the legacy
// mma.sync.m16n8k16 bf16 rate (the MMA the selected-attention kernels use), the
// ex2.approx rate (softmax exponentials) and, for a KV cache kept in page-locked host
// memory, the rates at which the SMs read that memory over the CPU-GPU link: a streaming
// read, the same random 4 KB-slice gather, and a copy-engine host-to-device copy.
// Standalone program; no part of the library.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <cuda_runtime.h>

__global__ void read_kernel(const uint4* __restrict__ p, size_t n, int iters, unsigned* out) {
  unsigned acc = 0;
  const size_t tid = blockIdx.x * (size_t)blockDim.x + threadIdx.x, stride = (size_t)gridDim.x * blockDim.x;
  for (int it = 0; it < iters; ++it)
    for (size_t i = tid; i < n; i += stride) {
      const uint4 v = __ldcg(p + i);
      acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
  out[tid] = acc;
}

__device__ __forceinline__ uint32_t mix(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

// Each warp streams `iters` random (K, V) slice pairs of 4 KB each (16 rows x 256 B)
// through a 2-stage cp.async ring of 8 KB stages, as the prefill kernel's warps do.
__global__ void __launch_bounds__(128) gather_kernel(const uint8_t* __restrict__ buf, uint32_t n_slices,
                                                     int iters) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t wbase = (uint32_t)__cvta_generic_to_shared(sm) + warp * 2 * 8192;
  const uint32_t gw = blockIdx.x * 4 + warp;
  auto issue = [&](int i) {
    const uint32_t sk = mix(gw * 7919u + i) % n_slices, sv = mix(gw * 104729u + i) % n_slices;
    const uint32_t dst = wbase + (i & 1) * 8192;
#pragma unroll
    for (int c = lane; c < 256; c += 32) {
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst + c * 16),
                   "l"(buf + (size_t)sk * 4096 + c * 16));
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst + 4096 + c * 16),
                   "l"(buf + (size_t)sv * 4096 + c * 16));
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  };
  issue(0);
  for (int i = 0; i < iters; ++i) {
    if (i + 1 < iters) issue(i + 1);
    else asm volatile("cp.async.commit_group;\n" ::: "memory");
    asm volatile("cp.async.wait_group 1;\n" ::: "memory");
    __syncwarp();
  }
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

__device__ __forceinline__ void mma(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void mma_kernel(float* out, int iters) {
  const uint32_t a[4] = {0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u};
  const uint32_t b = 0x3c003c00u;
  float c[8][4] = {};
  for (int i = 0; i < iters; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) mma(c[j], a, b, b);
  float s = 0.f;
  for (int j = 0; j < 8; ++j)
    for (int q = 0; q < 4; ++q) s += c[j][q];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void ex2_kernel(float* out, int iters) {
  float x[8];
  for (int j = 0; j < 8; ++j) x[j] = -0.001f * (threadIdx.x + j);
  for (int i = 0; i < iters; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float y;
      asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x[j]));
      x[j] = y - 1.0f;
    }
  float s = 0.f;
  for (int j = 0; j < 8; ++j) s += x[j];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

static float timed_ms(void (*launch)(void*), void* arg) {
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  launch(arg);  // warm-up
  cudaDeviceSynchronize();
  cudaEventRecord(a);
  launch(arg);
  cudaEventRecord(b);
  cudaEventSynchronize(b);
  float ms = 0.f;
  cudaEventElapsedTime(&ms, a, b);
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  return ms;
}

struct ReadArg { const uint4* p; size_t n; int iters; unsigned* out; int grid; };
static void launch_read(void* v) {
  ReadArg* r = static_cast<ReadArg*>(v);
  read_kernel<<<r->grid, 256>>>(r->p, r->n, r->iters, r->out);
}
struct GatherArg { const uint8_t* buf; uint32_t n_slices; int iters; int grid; };
static void launch_gather(void* v) {
  GatherArg* g = static_cast<GatherArg*>(v);
  gather_kernel<<<g->grid, 128, 2 * 4 * 8192>>>(g->buf, g->n_slices, g->iters);
}
struct ComputeArg { float* out; int iters; int grid; bool mma; };
static void launch_compute(void* v) {
  ComputeArg* c = static_cast<ComputeArg*>(v);
  if (c->mma) mma_kernel<<<c->grid, 256>>>(c->out, c->iters);
  else ex2_kernel<<<c->grid, 256>>>(c->out, c->iters);
}

int main() {
  int sms = 0, clk_khz = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, 0);
  const int grid = sms * 8;
  unsigned* out = nullptr;
  cudaMalloc(&out, (size_t)grid * 256 * 4);
  double bw[2] = {0, 0};
  const size_t mbs[2] = {64, 4096};  // L2-resident and HBM-sized buffers
  for (int t = 0; t < 2; ++t) {
    const size_t n = mbs[t] * (1u << 20) / 16;
    uint4* p = nullptr;
    if (cudaMalloc(&p, n * 16) != cudaSuccess) { printf("{\"error\": \"allocation\"}\n"); return 1; }
    cudaMemset(p, 1, n * 16);
    ReadArg r{p, n, t == 0 ? 20 : 2, out, grid};
    const float ms = timed_ms(launch_read, &r);
    bw[t] = (double)n * 16 * r.iters / (ms * 1e-3) / 1e9;
    cudaFree(p);
  }
  double gather = 0;
  {
    const size_t bytes = (size_t)32 << 20;  // L2 resident, like the benchmark's K and V
    uint8_t* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) { printf("{\"error\": \"allocation\"}\n"); return 1; }
    cudaMemset(p, 1, bytes);
    cudaFuncSetAttribute(gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * 4 * 8192);
    GatherArg g{p, (uint32_t)(bytes / 4096), 512, sms * 3};
    const float ms = timed_ms(launch_gather, &g);
    gather = (double)g.grid * 4 * g.iters * 8192.0 / (ms * 1e-3) / 1e9;
    cudaFree(p);
  }
  double c2c_read = 0, c2c_gather = 0, h2d_copy = 0;
  {
    const size_t bytes = (size_t)1 << 30;
    uint8_t* h = nullptr;
    uint8_t* d = nullptr;
    if (cudaHostAlloc(&h, bytes, cudaHostAllocMapped) != cudaSuccess || cudaMalloc(&d, bytes) != cudaSuccess) {
      printf("{\"error\": \"host allocation\"}\n");
      return 1;
    }
    memset(h, 1, bytes);
    uint8_t* hd = nullptr;
    cudaHostGetDevicePointer(reinterpret_cast<void**>(&hd), h, 0);
    ReadArg r{reinterpret_cast<const uint4*>(hd), bytes / 16, 1, out, grid};
    c2c_read = (double)bytes / (timed_ms(launch_read, &r) * 1e-3) / 1e9;
    GatherArg g{hd, (uint32_t)(bytes / 4096), 64, sms * 3};
    c2c_gather = (double)g.grid * 4 * g.iters * 8192.0 / (timed_ms(launch_gather, &g) * 1e-3) / 1e9;
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    cudaMemcpyAsync(d, h, bytes, cudaMemcpyHostToDevice);
    cudaEventRecord(a);
    cudaMemcpyAsync(d, h, bytes, cudaMemcpyHostToDevice);
    cudaEventRecord(b);
    cudaEventSynchronize(b);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, a, b);
    h2d_copy = (double)bytes / (ms * 1e-3) / 1e9;
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    cudaFree(d);
    cudaFreeHost(h);
  }
  float* fo = nullptr;
  cudaMalloc(&fo, (size_t)sms * 4 * 256 * 4);
  ComputeArg cm{fo, 4096, sms * 4, true};
  const float ms_mma = timed_ms(launch_compute, &cm);
  const double mma_tf = (double)cm.grid * 256 / 32 * cm.iters * 8 * 4096 / (ms_mma * 1e-3) / 1e12;
  ComputeArg ce{fo, 4096, sms * 4, false};
  const float ms_ex2 = timed_ms(launch_compute, &ce);
  const double ex2_rate = (double)ce.grid * 256 * ce.iters * 8 / (ms_ex2 * 1e-3);
  const cudaError_t e = cudaGetLastError();
  printf("{\"l2_read_gbs\": %.1f, \"l2_gather_gbs\": %.1f, \"hbm_read_gbs\": %.1f, "
         "\"mma_sync_bf16_tflops\": %.1f, \"ex2_per_sm_per_clk\": %.2f, \"c2c_read_gbs\": %.1f, "
         "\"c2c_gather_gbs\": %.1f, \"h2d_copy_gbs\": %.1f, \"sms\": %d, \"clock_mhz\": %.0f, "
         "\"error\": \"%s\"}\n",
         bw[0], gather, bw[1], mma_tf, ex2_rate / sms / (clk_khz * 1e3), c2c_read, c2c_gather, h2d_copy, sms,
         clk_khz / 1e3,
         e == cudaSuccess ? "" : cudaGetErrorString(e));
  cudaFree(out);
  cudaFree(fo);
  return e == cudaSuccess ? 0 : 1;
}
