// The streaming kernel's variants that cut the blocks of the partial last
// round into column parts, in a translation unit of their own (they compile
// in parallel with the others).

#include "mhc_stream_kernel.cuh"

namespace mhc {

void* stream_kernel_ptr_split(int form, int out, bool ms, int kcl) { return stream_kernel_ptr_t<2>(form, out, ms, kcl); }

}  // namespace mhc
