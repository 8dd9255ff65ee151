// sparse decode-attention kernel instantiations (head dim 64/128; a CTA takes at most 32
// query heads, so only the padded groups 8, 16 and 32 exist).
#include "launch.h"

namespace da {

template <int D, int GP>
static cudaError_t run_sparse(const Launch& L) {
    return launch_kernel(reinterpret_cast<const void*>(&decode_attn_kernel<kSparse, D, GP>),
                         Geometry<D, GP>::kSmemBytes, L);
}

cudaError_t launch_sparse(int D, int GP, const Launch& L) {
    if (D == 64) {
        switch (GP) {
            case 8: return run_sparse<64, 8>(L);
            case 16: return run_sparse<64, 16>(L);
            case 32: return run_sparse<64, 32>(L);
        }
    } else if (D == 128) {
        switch (GP) {
            case 8: return run_sparse<128, 8>(L);
            case 16: return run_sparse<128, 16>(L);
            case 32: return run_sparse<128, 32>(L);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace da
