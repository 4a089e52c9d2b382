// attention_mma_d64_l.cu -- instantiations of the paged decode attention
// kernel with tensor-core consumers: head_dim 64, 12 or 16 rows per
// kv-head (fewer rows take the next instance up).
#include "attention_kernel.cuh"

namespace pkv {
namespace attn {

KernelInfo kernel_mma_d64_l(int g, int hg) {
    if (g <= 12) return mma_by_heads<64, 12>(hg);
    if (g <= 16) return mma_by_heads<64, 16>(hg);
    return {nullptr, 0, nullptr, 0, nullptr};
}

}  // namespace attn
}  // namespace pkv
