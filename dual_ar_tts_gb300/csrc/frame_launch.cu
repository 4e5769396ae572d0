// Host side of the frame kernel: picks the kernel instance for a model's configuration, sizes
// the grid (one CTA per SM, cooperative) and launches it.
#include <cuda_runtime.h>

#include "s2_internal.h"

namespace s2 {

const void* frame_kernel_bf16_h128();
const void* frame_kernel_bf16_h64();
const void* frame_kernel_f32_h128();
const void* frame_kernel_f32_h64();
size_t frame_kernel_smem_bytes();

namespace {

__global__ void k_set_u32(unsigned* p, unsigned v) { *p = v; }

// bf16 weights run with an fp16 KV cache, fp32 weights with an fp32 cache; the head_dim of the
// Fast-AR transformer (equal to the Slow-AR one when there is a Slow-AR) selects the rest
const void* kernel_for(const Dims& d) {
  if (d.wdt == S2_BF16) return d.hdf == 128 ? frame_kernel_bf16_h128() : frame_kernel_bf16_h64();
  return d.hdf == 128 ? frame_kernel_f32_h128() : frame_kernel_f32_h64();
}

}  // namespace

int frame_kernel_grid(int device, int* grid_out) {
  const int smem = static_cast<int>(frame_kernel_smem_bytes());
  const void* all[4] = {frame_kernel_bf16_h128(), frame_kernel_bf16_h64(), frame_kernel_f32_h128(),
                        frame_kernel_f32_h64()};
  for (const void* k : all)
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return S2_ECUDA;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return S2_ECUDA;
  for (const void* k : all) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, smem) != cudaSuccess) return S2_ECUDA;
    if (per_sm < 1) return S2_ECUDA;
  }
  *grid_out = sms;  // one CTA per SM
  return S2_OK;
}

int launch_frames(const CallParams& cp, int grid, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the grid-barrier counter starts at cp.gbar_base (0 unless a test moves it near 2^32)
  if (cp.gbar_base == 0u) {
    if (cudaMemsetAsync(&cp.ctl->gbar, 0, sizeof(unsigned), s) != cudaSuccess) return S2_ECUDA;
  } else {
    k_set_u32<<<1, 1, 0, s>>>(&cp.ctl->gbar, cp.gbar_base);
    if (cudaGetLastError() != cudaSuccess) return S2_ECUDA;
  }
  void* args[] = {const_cast<CallParams*>(&cp)};
  const cudaError_t e = cudaLaunchCooperativeKernel(kernel_for(cp.d), dim3(grid), dim3(kThreads), args,
                                                    frame_kernel_smem_bytes(), s);
  return e == cudaSuccess ? S2_OK : S2_ECUDA;
}

size_t frame_kernel_smem() { return frame_kernel_smem_bytes(); }

}  // namespace s2
