// pa_decode_bf16.cu -- instantiations of the decode kernel for bf16 K/V.
#include "pkv_host.cuh"

namespace pkv {
int launch_decode_bf16(const DecodeLaunch &a) { return dispatch_decode<__nv_bfloat16>(a); }
}  // namespace pkv
