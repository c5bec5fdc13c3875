// kq_inst_3.cu -- kernels for ntok = 3 (see kq_launch.cuh).
#include "kq_launch.cuh"

KQ_DEFINE_INSTANCES(3)
