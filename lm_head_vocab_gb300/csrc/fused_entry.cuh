// Addresses of the staged-row kernel's instantiations.  Each (dtype, teacher,
// temperature) combination is instantiated in its own object file, compiled
// from fused_inst.cu, so that the library's translation units build in
// parallel; the host code reaches them only through these functions.
#pragma once

namespace lmloss {

// fused_kernel<BF16, KL, nt, stats, TAU> for a block of nt threads (128, 256,
// 512 or 1024), or null for any other nt.  stats selects the statistics-pass
// instantiation (no gradient, early buffer hand-off).
template <bool BF16, bool KL, bool TAU>
const void* fused_entry(int nt, bool stats);

extern template const void* fused_entry<true, false, false>(int, bool);
extern template const void* fused_entry<true, true, false>(int, bool);
extern template const void* fused_entry<true, true, true>(int, bool);
extern template const void* fused_entry<false, false, false>(int, bool);
extern template const void* fused_entry<false, true, false>(int, bool);
extern template const void* fused_entry<false, true, true>(int, bool);

}  // namespace lmloss
