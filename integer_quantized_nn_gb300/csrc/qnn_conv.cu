// qnn_conv.cu -- implicit-GEMM convolution (not yet implemented on the device).
#include <cuda_runtime.h>
#include "qnn_internal.h"

extern "C" size_t qnn_conv_packed_w_bytes(const qnn_conv_geom *g)
{
    (void)g;
    return 0;
}

extern "C" qnn_status qconv_prepack_w(const void *, qnn_dtype, const qnn_conv_geom *, void *, int32_t *,
                                      qnn_stream_t)
{
    return QNN_ERR_UNSUPPORTED;
}

extern "C" qnn_status qconv_u4s4(const void *, int32_t, const void *, const qnn_conv_geom *,
                                 const qnn_epilogue *, void *, int32_t *, qnn_stream_t)
{
    return QNN_ERR_UNSUPPORTED;
}

extern "C" qnn_status qconv_u8s8(const void *, int32_t, const void *, const qnn_conv_geom *,
                                 const qnn_epilogue *, void *, int32_t *, qnn_stream_t)
{
    return QNN_ERR_UNSUPPORTED;
}
