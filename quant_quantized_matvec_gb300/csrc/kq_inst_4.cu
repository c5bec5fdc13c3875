// kq_inst_4.cu -- kernels for ntok = 4 (see kq_launch.cuh).
#include "kq_launch.cuh"

KQ_DEFINE_INSTANCES(4)
