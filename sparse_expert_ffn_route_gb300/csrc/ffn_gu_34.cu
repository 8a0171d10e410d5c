// ffn_gu_34.cu -- instantiations of the expert-FFN kernel (gate/up, 3 or 4 chunks per lane).
#include "ffn_kernels.cuh"

namespace moe {

ffn_impl::Variant ffn_variant_gu_34(int nc, int tc)
{
    return nc == 3 ? ffn_impl::variant_nc<true, 3>(tc) : ffn_impl::variant_nc<true, 4>(tc);
}

}  // namespace moe
