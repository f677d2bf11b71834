// Launchers for 4-bit codes.
#define QMM_INST_BITS 4
#include "qmm_inst.cuh"
