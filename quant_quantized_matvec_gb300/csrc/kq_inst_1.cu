// kq_inst_1.cu -- kernels for ntok = 1 (see kq_launch.cuh).
#include "kq_launch.cuh"

KQ_DEFINE_INSTANCES(1)
