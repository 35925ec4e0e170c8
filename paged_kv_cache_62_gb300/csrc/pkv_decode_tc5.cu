// Instantiations of the query-split decode kernel on the 5th-generation tensor
// cores (tcgen05 products with tensor-memory accumulators: 128-row entries of
// 16 virtual-head blocks against 128-key tiles, long runs of new tokens in
// pkv_paged_attention), in a translation unit of their own so that they
// compile in parallel with the other kernel families.
#include "pkv_decode_kernel.cuh"

namespace pkv {

LaunchFn pick_decode_tc5(int D)
{
    if (D == 64) return launch_decode<64, 16, false, true, true>;
    if (D == 128) return launch_decode<128, 16, false, true, true>;
    return nullptr;
}

}  // namespace pkv
