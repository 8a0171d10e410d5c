// ffn_gu_78.cu -- instantiations of the expert-FFN kernel (gate/up, 7 or 8 chunks per lane).
#include "ffn_kernels.cuh"

namespace moe {

ffn_impl::Variant ffn_variant_gu_78(int nc, int tc)
{
    return nc == 7 ? ffn_impl::variant_nc<true, 7>(tc) : ffn_impl::variant_nc<true, 8>(tc);
}

}  // namespace moe
