// host_util.h -- host helpers shared by the library's C-ABI translation units
// (api.cu owns them): the per-thread error message, the driver entry points
// (tensor-map encoding, stream memory writes) and the default wait bound.
#pragma once

#include <cuda.h>

#include <cstdint>
#include <string>

namespace syn {

// Record `msg` as syn_last_error()'s text and return `code`.
int host_fail(int code, const std::string &msg);
// Resolve the driver entry points once; SYN_OK or SYN_ERR_CUDA.
int host_load_driver();
// 2-D tiled tensor map over a row-major matrix [rows, cols] of `esize`-byte
// elements, boxes of box_cols x box_rows.
int host_encode_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, uint64_t cols,
                   uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz);
// cuStreamWriteValue32 (the copy-engine backends' flag write).
CUresult host_write32(cudaStream_t st, uint32_t *addr, uint32_t value);
// SYN_TIMEOUT_NS from the environment, else 2 s.
uint64_t host_timeout_ns();

}  // namespace syn
