// Paged decode attention over an INT8 cache (dequantised as
// (x_q - zero_point) * scale, "cs336 lecture 10" Quantization).
#include "pa_internal.h"

namespace pa {

pa_status launch_decode_int8(const DecodeArgs&) {
    return fail(PA_ERR_UNSUPPORTED, "INT8 decode is not built yet");
}

}  // namespace pa
