// attention_mma_d128_s.cu -- instantiations of the paged decode attention
// kernel with tensor-core consumers: head_dim 128, 1, 4 or 8 rows per
// kv-head (fewer rows take the next instance up).
#include "attention_kernel.cuh"

namespace pkv {
namespace attn {

KernelInfo kernel_mma_d128_s(int g, int hg) {
    if (g <= 1) return mma_by_heads<128, 1>(hg);
    if (g <= 4) return mma_by_heads<128, 4>(hg);
    if (g <= 8) return mma_by_heads<128, 8>(hg);
    return {nullptr, 0, nullptr, 0, nullptr};
}

}  // namespace attn
}  // namespace pkv
