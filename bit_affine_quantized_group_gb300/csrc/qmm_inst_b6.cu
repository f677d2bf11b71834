// Launchers for 6-bit codes.
#define QMM_INST_BITS 6
#include "qmm_inst.cuh"
