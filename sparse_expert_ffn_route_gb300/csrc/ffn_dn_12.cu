// ffn_dn_12.cu -- instantiations of the expert-FFN kernel (down, 1 or 2 chunks per lane).
#include "ffn_kernels.cuh"

namespace moe {

ffn_impl::Variant ffn_variant_dn_12(int nc, int tc)
{
    return nc == 1 ? ffn_impl::variant_nc<false, 1>(tc) : ffn_impl::variant_nc<false, 2>(tc);
}

}  // namespace moe
