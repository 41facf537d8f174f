// ncbwd_ffma.cu -- instantiations of the CUDA-core non-causal backward launcher.
#include "noncausal_bwd_ffma.cuh"

namespace la {

#define LA_INST_NCB(T, D, M)                                                                      \
    template cudaError_t noncausal_backward<T, D, M>(const LaunchCtx&, const T*, const T*,       \
                                                     const T*, const T*, const T*, T*, T*, T*,   \
                                                     int, int);
#define LA_INST_NCB_T(T)                                                           \
    LA_INST_NCB(T, 32, 32) LA_INST_NCB(T, 32, 64) LA_INST_NCB(T, 32, 128)          \
    LA_INST_NCB(T, 64, 32) LA_INST_NCB(T, 64, 64) LA_INST_NCB(T, 64, 128)          \
    LA_INST_NCB(T, 128, 32) LA_INST_NCB(T, 128, 64) LA_INST_NCB(T, 128, 128)
LA_INST_NCB_T(float)
LA_INST_NCB_T(__nv_bfloat16)

}  // namespace la
