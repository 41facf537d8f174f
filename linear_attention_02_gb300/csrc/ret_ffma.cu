// ret_ffma.cu -- instantiations of the CUDA-core retention forward launcher.
#include "retention_ffma.cuh"

namespace la {

#define LA_INST_RET(T, D, M)                                                                     \
    template cudaError_t retention_forward<T, D, M>(const LaunchCtx&, const T*, const T*,       \
                                                    const T*, T*, const float*, const float*,   \
                                                    int, int, int, const float*, float*);
#define LA_INST_RET_T(T)                                                           \
    LA_INST_RET(T, 32, 32) LA_INST_RET(T, 32, 64) LA_INST_RET(T, 32, 128)          \
    LA_INST_RET(T, 64, 32) LA_INST_RET(T, 64, 64) LA_INST_RET(T, 64, 128)          \
    LA_INST_RET(T, 128, 32) LA_INST_RET(T, 128, 64) LA_INST_RET(T, 128, 128)
LA_INST_RET_T(float)
LA_INST_RET_T(__nv_bfloat16)

}  // namespace la
