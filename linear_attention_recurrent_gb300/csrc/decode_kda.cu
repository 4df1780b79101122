// decode_kda.cu -- KDA instantiation of the decode kernel (one translation unit
// per form so the build compiles them in parallel).
#include "decode_kernel.cuh"
#include "decode_kv_kernel.cuh"

namespace lar {

lar_status launch_kda(const DecodeParams& p, void* stream) {
    return p.state_kv ? launch_form_kv<FORM_KDA>(p, stream) : launch_form<FORM_KDA>(p, stream);
}

}  // namespace lar
