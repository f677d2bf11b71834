// Launchers for 3-bit codes.
#define QMM_INST_BITS 3
#include "qmm_inst.cuh"
