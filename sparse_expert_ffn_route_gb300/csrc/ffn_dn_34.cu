// ffn_dn_34.cu -- instantiations of the expert-FFN kernel (down, 3 or 4 chunks per lane).
#include "ffn_kernels.cuh"

namespace moe {

ffn_impl::Variant ffn_variant_dn_34(int nc, int tc)
{
    return nc == 3 ? ffn_impl::variant_nc<false, 3>(tc) : ffn_impl::variant_nc<false, 4>(tc);
}

}  // namespace moe
