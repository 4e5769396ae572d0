// Codec quantizer decode, lookup-and-sum part (s2.cpp analysis ch.02 §3.5): for every frame, the
// rows its codes select in the semantic and residual VQ codebooks, summed in codebook order.
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"
#include "s2_internal.h"

namespace s2 {
namespace {

constexpr int kMaxQuantizers = 16;

struct QuantizerTable {
  const uint16_t* q[kMaxQuantizers];
};

// one CTA per frame; thread t sums 8-element groups of the latent row (16-byte loads)
__global__ void __launch_bounds__(256) k_codec_latent(QuantizerTable tab, int ncb, int cbs, int dim, int n_frames,
                                                      const int32_t* __restrict__ codes, float* __restrict__ latent,
                                                      int32_t* status) {
  __shared__ int code[kMaxQuantizers];
  const int f = blockIdx.x;
  if (threadIdx.x < ncb) {
    int c = codes[static_cast<size_t>(threadIdx.x) * n_frames + f];
    if (c < 0 || c >= cbs) {
      if (status) atomicCAS(status, 0, S2_EINVAL);
      c = -1;
    }
    code[threadIdx.x] = c;
  }
  __syncthreads();
  float* out = latent + static_cast<size_t>(f) * dim;
  for (int g = threadIdx.x; g < dim / 8; g += blockDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int cb = 0; cb < ncb; ++cb) {
      if (code[cb] < 0) continue;
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(tab.q[cb] + static_cast<size_t>(code[cb]) * dim) + g);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[2 * j] = __fadd_rn(acc[2 * j], bf16lo(w[j]));
        acc[2 * j + 1] = __fadd_rn(acc[2 * j + 1], bf16hi(w[j]));
      }
    }
    float4* o4 = reinterpret_cast<float4*>(out + 8 * g);
    o4[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o4[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

}  // namespace
}  // namespace s2

using namespace s2;

extern "C" int s2_codec_latent(int ncb, int cbs, int dim, const void* const* quantizers, int n_frames,
                               const int32_t* codes, float* latent, int32_t* status, CUstream_st* stream) {
  if (ncb < 1 || ncb > kMaxQuantizers || cbs < 1 || dim < 8 || dim % 8 != 0 || n_frames < 1 || !quantizers ||
      !codes || !latent)
    return S2_EINVAL;
  if (reinterpret_cast<uintptr_t>(latent) % 16 != 0) return S2_EINVAL;
  QuantizerTable tab{};
  for (int i = 0; i < ncb; ++i) {
    if (!quantizers[i] || reinterpret_cast<uintptr_t>(quantizers[i]) % 16 != 0) return S2_EINVAL;
    tab.q[i] = static_cast<const uint16_t*>(quantizers[i]);
  }
  k_codec_latent<<<n_frames, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(tab, ncb, cbs, dim, n_frames, codes,
                                                                               latent, status);
  return cudaGetLastError() == cudaSuccess ? S2_OK : S2_ECUDA;
}

extern "C" int s2_quantize_e4m3(const void* w, long long rows, int cols, uint8_t* codes, float* scales,
                                CUstream_st* stream) {
  if (!w || !codes || !scales || rows < 1 || cols < 1) return S2_EINVAL;
  if (reinterpret_cast<uintptr_t>(w) % 2 != 0 || reinterpret_cast<uintptr_t>(scales) % 4 != 0) return S2_EINVAL;
  return quantize_e4m3(w, rows, cols, codes, scales, stream) == 0 ? S2_OK : S2_ECUDA;
}
