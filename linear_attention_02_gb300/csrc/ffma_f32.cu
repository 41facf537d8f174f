// ffma_f32.cu -- instantiations of the CUDA-core causal and non-causal launchers for float.
#include "noncausal_ffma.cuh"

namespace la {

#define LA_INST(T, D, M)                                                                        \
    template cudaError_t causal_forward<T, D, M>(const LaunchCtx&, const T*, const T*, const T*, \
                                                 T*, int, int, const float*, const float*,     \
                                                 float*, float*, float*);                      \
    template cudaError_t causal_backward<T, D, M>(const LaunchCtx&, const T*, const T*,        \
                                                  const T*, const T*, const T*, T*, T*, T*,    \
                                                  int, int);                                   \
    template cudaError_t noncausal_forward<T, D, M>(const LaunchCtx&, const T*, const T*,      \
                                                    const T*, T*, int, int);
LA_INST(float, 32, 32) LA_INST(float, 32, 64) LA_INST(float, 32, 128)
LA_INST(float, 64, 32) LA_INST(float, 64, 64) LA_INST(float, 64, 128)
LA_INST(float, 128, 32) LA_INST(float, 128, 64) LA_INST(float, 128, 128)

}  // namespace la
