// ffn_dn_56.cu -- instantiations of the expert-FFN kernel (down, 5 or 6 chunks per lane).
#include "ffn_kernels.cuh"

namespace moe {

ffn_impl::Variant ffn_variant_dn_56(int nc, int tc)
{
    return nc == 5 ? ffn_impl::variant_nc<false, 5>(tc) : ffn_impl::variant_nc<false, 6>(tc);
}

}  // namespace moe
