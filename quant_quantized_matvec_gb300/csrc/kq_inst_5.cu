// kq_inst_5.cu -- kernels for ntok = 5 (see kq_launch.cuh).
#include "kq_launch.cuh"

KQ_DEFINE_INSTANCES(5)
