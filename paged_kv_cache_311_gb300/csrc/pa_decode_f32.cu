// pa_decode_f32.cu -- instantiations of the decode kernel for f32 K/V.
#include "pkv_host.cuh"

namespace pkv {
int launch_decode_f32(const DecodeLaunch &a) { return dispatch_decode<float>(a); }
}  // namespace pkv
