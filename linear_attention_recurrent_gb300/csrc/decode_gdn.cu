// decode_gdn.cu -- GDN instantiation of the decode kernel (one translation unit
// per form so the build compiles them in parallel).
#include "decode_kernel.cuh"

namespace lar {

lar_status launch_gdn(const DecodeParams& p, void* stream) { return launch_form<FORM_GDN>(p, stream); }

}  // namespace lar
