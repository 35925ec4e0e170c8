// Instantiations of the query-split decode kernel (bf16 caches; the CTA's
// warps share every K/V tile of one kv head, each with its own queries filling
// both 8-row halves of the MMA tile: long runs of new tokens in
// pkv_paged_attention), in a translation unit of their own so that they
// compile in parallel with the other kernel families.  A warp holds
// max(1, 16 / gq) queries of gq heads: G = 16, 15, 14 or 12 virtual heads.
#include "pkv_decode_kernel.cuh"

namespace pkv {

template <int D>
static LaunchFn pick_qs(int G)
{
    switch (G) {
    case 12: return launch_decode<D, 12, false, true>;
    case 14: return launch_decode<D, 14, false, true>;
    case 15: return launch_decode<D, 15, false, true>;
    case 16: return launch_decode<D, 16, false, true>;
    default: return nullptr;
    }
}

LaunchFn pick_decode_qs(int D, int G)
{
    if (D == 64) return pick_qs<64>(G);
    if (D == 128) return pick_qs<128>(G);
    return nullptr;
}

}  // namespace pkv
