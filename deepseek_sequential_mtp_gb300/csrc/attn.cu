#include "common.cuh"
MTP_DEFINE_ERROR_WORD(mtp_take_errors_attn)
