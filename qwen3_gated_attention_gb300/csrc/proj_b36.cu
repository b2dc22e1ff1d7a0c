// proj_b36.cu -- 3- and 6-bit instantiations of the projection kernel.
#include "proj_inst.cuh"
GATTN_PROJ_INSTANCE(3)
GATTN_PROJ_INSTANCE(6)
