// decode_gdn.cu -- GDN instantiation of the decode kernel (one translation unit
// per form so the build compiles them in parallel).
#include "decode_kernel.cuh"
#include "decode_kv_kernel.cuh"

namespace lar {

lar_status launch_gdn(const DecodeParams& p, void* stream) {
    return p.state_kv ? launch_form_kv<FORM_GDN>(p, stream) : launch_form<FORM_GDN>(p, stream);
}

}  // namespace lar
