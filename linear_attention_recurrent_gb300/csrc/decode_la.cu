// decode_la.cu -- LA instantiation of the decode kernel (one translation unit
// per form so the build compiles them in parallel).
#include "decode_kernel.cuh"

namespace lar {

lar_status launch_la(const DecodeParams& p, void* stream) { return launch_form<FORM_LA>(p, stream); }

}  // namespace lar
