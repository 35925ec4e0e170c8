// Instantiations of the regular decode kernel (bf16 caches) for 9 to 16
// virtual heads per kv head -- several new tokens per sequence whose
// (query, head) pairs fill both 8-row halves of the MMA tile -- in a
// translation unit of their own so that they compile in parallel with the
// other kernel families.
#include "pkv_decode_kernel.cuh"

namespace pkv {

template <int D>
static LaunchFn pick_wide(int G)
{
    switch (G) {
    case 9: return launch_decode<D, 9, false, false>;
    case 10: return launch_decode<D, 10, false, false>;
    case 11: return launch_decode<D, 11, false, false>;
    case 12: return launch_decode<D, 12, false, false>;
    case 13: return launch_decode<D, 13, false, false>;
    case 14: return launch_decode<D, 14, false, false>;
    case 15: return launch_decode<D, 15, false, false>;
    case 16: return launch_decode<D, 16, false, false>;
    default: return nullptr;
    }
}

LaunchFn pick_decode_wide(int D, int G)
{
    if (D == 64) return pick_wide<64>(G);
    if (D == 128) return pick_wide<128>(G);
    return nullptr;
}

}  // namespace pkv
