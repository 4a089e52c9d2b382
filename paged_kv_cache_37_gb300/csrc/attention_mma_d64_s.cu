// attention_mma_d64_s.cu -- instantiations of the paged decode attention
// kernel with tensor-core consumers: head_dim 64, 1, 4 or 8 rows per
// kv-head (fewer rows take the next instance up).
#include "attention_kernel.cuh"

namespace pkv {
namespace attn {

KernelInfo kernel_mma_d64_s(int g, int hg) {
    if (g <= 1) return mma_by_heads<64, 1>(hg);
    if (g <= 4) return mma_by_heads<64, 4>(hg);
    if (g <= 8) return mma_by_heads<64, 8>(hg);
    return {nullptr, 0, nullptr, 0, nullptr};
}

}  // namespace attn
}  // namespace pkv
