// Kernel instantiations for f32 elements, conv width 4.
#define CV_INST_B uint32_t
#define CV_INST_W 4
#define CV_INST_MAXT 8
#define CV_INST_NAME kernels_f32_w4
#include "cv_inst.cuh"
