// decode_kda.cu -- KDA instantiation of the decode kernel (one translation unit
// per form so the build compiles them in parallel).
#include "decode_kernel.cuh"

namespace lar {

lar_status launch_kda(const DecodeParams& p, void* stream) { return launch_form<FORM_KDA>(p, stream); }

}  // namespace lar
