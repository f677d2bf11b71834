// Launchers for 5-bit codes.
#define QMM_INST_BITS 5
#include "qmm_inst.cuh"
