// Launchers for 8-bit codes.
#define QMM_INST_BITS 8
#include "qmm_inst.cuh"
