// Instantiations of the decode kernel for E4M3 (fp8) caches, in a translation
// unit of their own so that they compile in parallel with the bf16 ones.
#include "pkv_decode_kernel.cuh"

namespace pkv {

LaunchFn pick_decode_fp8(int D, int G)
{
    if (D == 64) return pick_group<64, true, false>(G);
    if (D == 128) return pick_group<128, true, false>(G);
    return nullptr;
}

}  // namespace pkv
