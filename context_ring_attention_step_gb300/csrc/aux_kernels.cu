// aux_kernels.cu -- the HBM-bound passes around the ring steps:
//   * cast of the fp32 running output to the bf16 result (forward finalise);
//   * backward preprocess: Delta = rowsum(dO * O) with 8-lane shuffle
//     reductions, and LSE rescaled to log2 units for the exp2-based recompute;
//     both stored negated (-Delta, -LSE log2e), the form the backward kernels
//     add with packed fp32 arithmetic.
#include <cuda_bf16.h>

#include <algorithm>

#include "ring_attn_internal.h"
#include "tc.cuh"

namespace ra {
namespace {

// Failure-detection self-test: one thread waits, with a short limit, on an
// mbarrier that nothing ever arrives on, through the same bounded wait the
// ring kernels use; it gives up, records `site` in the status word and the
// kernel returns.
__global__ void wait_timeout_probe_kernel(int* status, uint64_t limit_ns, int site) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const Abort ab{&abort_flag, status};
    (void)mbar_wait(smem_u32(&bar), 0, ab, site, limit_ns);
  }
}

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// n8 = number of 8-element groups
// Workspace set-up without the copy engines: zero the status header and copy
// up to two work lists from mapped pinned host memory (read over the host
// link by the SMs).  Sizes are multiples of 16 bytes.
__global__ void ws_init_kernel(uint4* __restrict__ header, int header16, const uint4* __restrict__ src0,
                               uint4* __restrict__ dst0, size_t n0, const uint4* __restrict__ src1,
                               uint4* __restrict__ dst1, size_t n1) {
  const size_t tid = blockIdx.x * (size_t)blockDim.x + threadIdx.x, stride = (size_t)gridDim.x * blockDim.x;
  if (tid < (size_t)header16) header[tid] = make_uint4(0u, 0u, 0u, 0u);
  for (size_t i = tid; i < n0; i += stride) dst0[i] = src0[i];
  for (size_t i = tid; i < n1; i += stride) dst1[i] = src1[i];
}

__global__ void cast_bf16_kernel(const float4* __restrict__ src, uint4* __restrict__ dst, size_t n8) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = __ldcs(src + 2 * i);
    const float4 b = __ldcs(src + 2 * i + 1);
    uint4 o;
    o.x = pack2(a.x, a.y);
    o.y = pack2(a.z, a.w);
    o.z = pack2(b.x, b.y);
    o.w = pack2(b.z, b.w);
    __stcs(dst + i, o);
  }
}

__device__ __forceinline__ void load8(const void* base, size_t elem, bool fp32, float (&x)[8]) {
  if (fp32) {
    const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + elem);
    const float4 a = p[0], b = p[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(base) + elem);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}

// 8 lanes per (t, h) row; each lane covers D/8 consecutive elements.
template <int D>
__global__ void bwd_preprocess_kernel(const void* __restrict__ o, int o_fp32, const void* __restrict__ dout,
                                      const float* __restrict__ lse, float* __restrict__ delta,
                                      float* __restrict__ lse2, int T, int64_t pitch, int Hq, float scale) {
  const long long rows = (long long)T * Hq;
  const long long row = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 3;
  const int sub = threadIdx.x & 7;
  float acc = 0.f;
  if (row < rows) {
    constexpr int E = D / 8;
#pragma unroll
    for (int e = 0; e < E; e += 8) {
      const size_t elem = (size_t)row * D + sub * E + e;
      float a[8], b[8];
      load8(dout, elem, false, a);
      load8(o, elem, o_fp32 != 0, b);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(a[i], b[i], acc);
    }
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  if (row < rows && sub == 0) {
    const int t = (int)(row / Hq), h = (int)(row % Hq);
    const size_t idx = (size_t)h * pitch + t;
    delta[idx] = -acc * scale;
    lse2[idx] = -lse[(size_t)h * T + t] * kLog2e;
  }
}

}  // namespace

cudaError_t launch_cast_bf16(const float* src, void* dst, size_t n, cudaStream_t stream) {
  const size_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  const int threads = 256;
  const size_t want = (n8 + threads - 1) / threads;
  const unsigned blocks = (unsigned)(want < 152 * 16 ? want : 152 * 16);
  cast_bf16_kernel<<<blocks, threads, 0, stream>>>(reinterpret_cast<const float4*>(src),
                                                    reinterpret_cast<uint4*>(dst), n8);
  return cudaGetLastError();
}

cudaError_t launch_ws_init(void* header, size_t header_bytes, const void* src0, void* dst0, size_t bytes0,
                          const void* src1, void* dst1, size_t bytes1, cudaStream_t stream) {
  const size_t n0 = bytes0 / 16, n1 = bytes1 / 16, most = std::max(std::max(n0, n1), header_bytes / 16);
  const int threads = 256;
  const unsigned blocks = (unsigned)std::min<size_t>(std::max<size_t>((most + threads - 1) / threads, 1), 152);
  ws_init_kernel<<<blocks, threads, 0, stream>>>(reinterpret_cast<uint4*>(header), (int)(header_bytes / 16),
                                                  reinterpret_cast<const uint4*>(src0), reinterpret_cast<uint4*>(dst0),
                                                  n0, reinterpret_cast<const uint4*>(src1),
                                                  reinterpret_cast<uint4*>(dst1), n1);
  return cudaGetLastError();
}

cudaError_t launch_bwd_preprocess(const void* o, int o_is_fp32, const void* dout, const float* lse, float* delta,
                                  float* lse2, int T, int64_t pitch, int Hq, int D, float scale,
                                  cudaStream_t stream) {
  const long long threads_needed = (long long)T * Hq * 8;
  if (threads_needed == 0) return cudaSuccess;
  const int threads = 256;
  const unsigned blocks = (unsigned)((threads_needed + threads - 1) / threads);
  if (D == 128)
    bwd_preprocess_kernel<128><<<blocks, threads, 0, stream>>>(o, o_is_fp32, dout, lse, delta, lse2, T, pitch, Hq, scale);
  else if (D == 64)
    bwd_preprocess_kernel<64><<<blocks, threads, 0, stream>>>(o, o_is_fp32, dout, lse, delta, lse2, T, pitch, Hq, scale);
  else if (D == 256)
    bwd_preprocess_kernel<256><<<blocks, threads, 0, stream>>>(o, o_is_fp32, dout, lse, delta, lse2, T, pitch, Hq, scale);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_probe(int* status, uint64_t limit_ns, int site, cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns, site);
  return cudaGetLastError();
}

}  // namespace ra
