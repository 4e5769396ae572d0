// Frame kernel instance: fp32 weights, fp32 KV cache, head_dim 64.
#include "frame_kernel.cuh"

namespace s2 {
const void* frame_kernel_f32_h64() { return reinterpret_cast<const void*>(&frame_kernel<Cfg<false, 64>>); }
}  // namespace s2
