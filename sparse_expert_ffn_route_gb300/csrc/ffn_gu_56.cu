// ffn_gu_56.cu -- instantiations of the expert-FFN kernel (gate/up, 5 or 6 chunks per lane).
#include "ffn_kernels.cuh"

namespace moe {

ffn_impl::Variant ffn_variant_gu_56(int nc, int tc)
{
    return nc == 5 ? ffn_impl::variant_nc<true, 5>(tc) : ffn_impl::variant_nc<true, 6>(tc);
}

}  // namespace moe
