// Frame kernel instance: bf16 weights, fp16 KV cache, head_dim 64.
#include "frame_kernel.cuh"

namespace s2 {
const void* frame_kernel_bf16_h64() { return reinterpret_cast<const void*>(&frame_kernel<Cfg<true, 64>>); }
}  // namespace s2
