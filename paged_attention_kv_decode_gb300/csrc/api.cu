// Library-wide host code: error messages, TMA descriptor encoding, status.
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdio.h>

#include <mutex>

#include "../../include/metis_attn.h"
#include "host.h"

namespace metis {

static thread_local char g_last_error[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { g_last_error[0] = '\0'; }

int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(METIS_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return METIS_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;
static cudaError_t g_encode_err = cudaSuccess;

static void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

int encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return fail(METIS_E_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(g_encode_err));
  cuuint64_t d[5];
  cuuint64_t st[4];
  cuuint32_t bx[5];
  cuuint32_t es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  CUresult r = g_encode(map, dtype, rank, const_cast<void*>(base), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(METIS_E_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return METIS_OK;
}

int set_max_dynamic_smem(const void* func, int bytes, int* done_mask) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(METIS_E_CUDA, "cudaGetDevice failed");
  const int bit = 1 << (dev & 31);
  if (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit) return METIS_OK;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return fail(METIS_E_CUDA, "cudaFuncSetAttribute(%d bytes): %s", bytes, cudaGetErrorString(e));
  __atomic_fetch_or(done_mask, bit, __ATOMIC_ACQ_REL);
  return METIS_OK;
}

}  // namespace metis

extern "C" const char* metis_last_error(void) { return metis::g_last_error; }

extern "C" int metis_version(void) { return 100; }

extern "C" int metis_read_status(uint32_t* status_out, int clear) {
  metis::clear_error();
  if (!status_out) return metis::fail(METIS_E_NULL, "status_out is NULL");
  uint32_t bits = 0;
  int rc = metis::decode_status(&bits, clear);
  if (rc) return rc;
  rc = metis::prefill_status(&bits, clear);
  if (rc) return rc;
  rc = metis::mla_status(&bits, clear);
  if (rc) return rc;
  rc = metis::cache_status(&bits, clear);
  if (rc) return rc;
  rc = metis::prefix_status(&bits, clear);
  if (rc) return rc;
  *status_out = bits;
  return METIS_OK;
}
