// Instantiations of the query-split decode kernel (bf16 caches; the CTA's
// warps share every K/V tile of one kv head, each with its own queries: long
// runs of new tokens in pkv_paged_attention), in a translation unit of their
// own so that they compile in parallel with the other kernel families.
#include "pkv_decode_kernel.cuh"

namespace pkv {

LaunchFn pick_decode_qs(int D, int G)
{
    if (D == 64) return pick_group<64, false, true>(G);
    if (D == 128) return pick_group<128, false, true>(G);
    return nullptr;
}

}  // namespace pkv
