// Launchers for 2-bit codes.
#define QMM_INST_BITS 2
#include "qmm_inst.cuh"
