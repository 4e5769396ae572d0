// The S2 sampler on caller logits rows: the draw routine the decode engines run (sampler.cuh), one
// CTA of 256 threads per row.  ch.06 "Fast-AR codebook decoding and the generation main loop" §5
// (the draw, min_tokens masking of im_end) and the Mizuoto "Fish Speech" engine page (top-k fixed at
// 30, argmax(probs / -log u)).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "ptx.cuh"
#include "s2_internal.h"
#include "sampler.cuh"

namespace s2 {
namespace {

static_assert(sizeof(SampScratch) <= 48 * 1024, "sampler scratch within the default shared memory");

__global__ void __launch_bounds__(kConsumers) k_draw_rows(const Dims d, const float* __restrict__ logits, int n,
                                                          int is_main, int block_end, float temperature, float top_p,
                                                          const float* __restrict__ expo, int32_t* __restrict__ out) {
  extern __shared__ __align__(16) unsigned char smraw[];
  SampScratch& W = *reinterpret_cast<SampScratch*>(smraw);
  const size_t r = blockIdx.x;
  const int v = draw(d, W, logits + r * n, n, is_main != 0, block_end != 0, temperature, top_p, expo + r * kTopK);
  if (threadIdx.x == 0) out[r] = v;
}

}  // namespace
}  // namespace s2

using namespace s2;

extern "C" int s2_draw(int rows, const float* logits, int n, int sem_begin, int im_end, int block_end,
                       float temperature, float top_p, const float* expo, int32_t* out, CUstream_st* stream) {
  if (rows < 1 || n < 1 || n > kSampPer * kConsumers || !logits || !expo || !out) return S2_EINVAL;
  if (reinterpret_cast<uintptr_t>(logits) % 4 != 0 || reinterpret_cast<uintptr_t>(expo) % 4 != 0 ||
      reinterpret_cast<uintptr_t>(out) % 4 != 0)
    return S2_EINVAL;
  if (!std::isfinite(temperature) || temperature <= 0.f || !std::isfinite(top_p)) return S2_EINVAL;
  const bool is_main = sem_begin >= 0;
  if (is_main && n < 2) return S2_EINVAL;
  // the draw maps entry i to its id through these fields alone
  Dims d{};
  d.sem_lo = is_main ? sem_begin : 0;
  d.cbs = is_main ? n - 1 : n;
  d.sem_hi = d.sem_lo + d.cbs - 1;
  d.im_end = im_end;
  d.A = n;
  k_draw_rows<<<rows, kConsumers, sizeof(SampScratch), reinterpret_cast<cudaStream_t>(stream)>>>(
      d, logits, n, is_main ? 1 : 0, block_end ? 1 : 0, temperature, top_p, expo, out);
  return cudaGetLastError() == cudaSuccess ? S2_OK : S2_ECUDA;
}
