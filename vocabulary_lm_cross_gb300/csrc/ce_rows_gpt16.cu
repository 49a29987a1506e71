// ce_rows_gpt16.cu -- instantiations of the row kernel holding up to 16
// granules (16-byte units) of its row slice per consumer thread.
#include "ce_rows.cuh"

VLMCE_DEFINE_ROWS_KERNEL_GETTER(16)
