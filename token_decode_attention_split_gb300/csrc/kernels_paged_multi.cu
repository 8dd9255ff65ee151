// paged decode-attention kernel instantiations for units of kh > 1 adjacent KV heads (head dim
// 64/128, padded group 8/16/32/64, and the warp-per-KV-head column layout for 16-column units).
#include "launch.h"

namespace da {

template <int D, int GP, int GW = GP>
static cudaError_t run_paged(const Launch& L) {
    return launch_kernel(reinterpret_cast<const void*>(&decode_attn_kernel<kPaged, D, GP, GW, true>),
                         Geometry<D, GP>::kSmemBytes, L);
}

cudaError_t launch_paged_multi(int D, int GP, bool warp_head, const Launch& L) {
    if (warp_head) {
        if (GP != 16) return cudaErrorInvalidValue;
        return D == 64 ? run_paged<64, 16, 8>(L) : D == 128 ? run_paged<128, 16, 8>(L)
                                                           : cudaErrorInvalidValue;
    }
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
