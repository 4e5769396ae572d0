// Frame kernel instance: fp32 weights, fp32 KV cache, head_dim 128.
#include "frame_kernel.cuh"

namespace s2 {
const void* frame_kernel_f32_h128() { return reinterpret_cast<const void*>(&frame_kernel<Cfg<false, 128>>); }
}  // namespace s2
