// Frame kernel instance: bf16 weights, fp16 KV cache, head_dim 128 (the S2-Pro shapes).
#include "frame_kernel.cuh"

namespace s2 {
const void* frame_kernel_bf16_h128() { return reinterpret_cast<const void*>(&frame_kernel<Cfg<true, 128>>); }
}  // namespace s2

namespace s2 {
size_t frame_kernel_smem_bytes() { return sizeof(Smem); }
}  // namespace s2
