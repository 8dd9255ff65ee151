// paged decode-attention kernel instantiations for units of one KV head (head dim 64/128, padded
// group 8/16/32/64): every consumer mask is a compile-time constant.
#include "launch.h"

namespace da {

template <int D, int GP>
static cudaError_t run_paged(const Launch& L) {
    return launch_kernel(reinterpret_cast<const void*>(&decode_attn_kernel<kPaged, D, GP, GP, false>),
                         Geometry<D, GP>::kSmemBytes, L);
}

cudaError_t launch_paged_single(int D, int GP, const Launch& L) {
    if (D == 64) {
        switch (GP) {
            case 8: return run_paged<64, 8>(L);
            case 16: return run_paged<64, 16>(L);
            case 32: return run_paged<64, 32>(L);
            case 64: return run_paged<64, 64>(L);
        }
    } else if (D == 128) {
        switch (GP) {
            case 8: return run_paged<128, 8>(L);
            case 16: return run_paged<128, 16>(L);
            case 32: return run_paged<128, 32>(L);
            case 64: return run_paged<128, 64>(L);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace da
