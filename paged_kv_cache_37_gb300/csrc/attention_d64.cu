// attention_d64.cu -- instantiations of the paged decode attention kernel
// for head_dim 64: 1..8 q-heads per kv-head, 1, 2 or 4 kv-heads per item.
#include "attention_kernel.cuh"

namespace pkv {
namespace attn {
namespace {

template <int G, int HG>
KernelInfo info() {
    if constexpr (RegisterCap<64, G, HG>::k128)
        return {paged_decode_kernel_r128<64, G, HG>, sizeof(Smem<64, G, HG>), merge_kernel<64, G, HG>, G,
                paged_decode_kernel_r128<64, G, HG>};
    else
        return {paged_decode_kernel<64, G, HG>, sizeof(Smem<64, G, HG>), merge_kernel<64, G, HG>, G,
                paged_decode_kernel<64, G, HG>};
}

template <int HG>
KernelInfo by_group(int g) {
    switch (g) {
        case 1: return info<1, HG>();
        case 2: return info<2, HG>();
        case 3: return info<3, HG>();
        case 4: return info<4, HG>();
        case 5: return info<5, HG>();
        case 6: return info<6, HG>();
        case 7: return info<7, HG>();
        case 8: return info<8, HG>();
        default: return {nullptr, 0, nullptr, 0, nullptr};
    }
}

}  // namespace

KernelInfo kernel_d64(int g, int hg) {
    switch (hg) {
        case 1: return by_group<1>(g);
        case 2: return by_group<2>(g);
        case 4: return by_group<4>(g);
        default: return {nullptr, 0, nullptr, 0, nullptr};
    }
}

}  // namespace attn
}  // namespace pkv
