// Instantiations of the staged-row kernel for one (dtype, teacher, temperature)
// combination, chosen by LMLOSS_FUSED_VARIANT (0..5) when this file is compiled;
// the library links the six objects.
#include "kernels.cuh"
#include "fused_entry.cuh"

#ifndef LMLOSS_FUSED_VARIANT
#error "compile with -DLMLOSS_FUSED_VARIANT=0..5"
#endif

namespace lmloss {

template <bool BF16, bool KL, bool TAU>
const void* fused_entry(int nt, bool stats)
{
    switch (nt) {
    case 128:
        return stats ? reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 128, true, TAU>)
                     : reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 128, false, TAU>);
    case 256:
        return stats ? reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 256, true, TAU>)
                     : reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 256, false, TAU>);
    case 512:
        return stats ? reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 512, true, TAU>)
                     : reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 512, false, TAU>);
    case 1024:
        return stats ? reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 1024, true, TAU>)
                     : reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 1024, false, TAU>);
    default:
        return nullptr;
    }
}

#if LMLOSS_FUSED_VARIANT == 0
template const void* fused_entry<true, false, false>(int, bool);
#elif LMLOSS_FUSED_VARIANT == 1
template const void* fused_entry<true, true, false>(int, bool);
#elif LMLOSS_FUSED_VARIANT == 2
template const void* fused_entry<true, true, true>(int, bool);
#elif LMLOSS_FUSED_VARIANT == 3
template const void* fused_entry<false, false, false>(int, bool);
#elif LMLOSS_FUSED_VARIANT == 4
template const void* fused_entry<false, true, false>(int, bool);
#elif LMLOSS_FUSED_VARIANT == 5
template const void* fused_entry<false, true, true>(int, bool);
#else
#error "LMLOSS_FUSED_VARIANT must be 0..5"
#endif

}  // namespace lmloss
