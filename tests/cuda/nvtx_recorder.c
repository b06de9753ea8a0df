/*
 * A minimal NVTX injection library for tests: NVTX v3 loads the library
 * named by NVTX_INJECTION64_PATH at a process's first NVTX call and calls
 * its InitializeInjectionNvtx2, which here replaces the core RangePushA and
 * RangePop entries so that every range opened or closed is appended to the
 * file named by OB_NVTX_LOG ("push <name>" / "pop" lines).  Host code only;
 * used by tests/test_nvtx_ranges.py on the CPU.
 */
#include <stdio.h>
#include <stdlib.h>

#include <nvtx3/nvToolsExt.h>

static FILE* g_log;

static int record_push(const char* message) {
  if (g_log) {
    fprintf(g_log, "push %s\n", message ? message : "");
    fflush(g_log);
  }
  return 0;
}

static int record_pop(void) {
  if (g_log) {
    fprintf(g_log, "pop\n");
    fflush(g_log);
  }
  return 0;
}

int InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_export_table) {
  const NvtxExportTableCallbacks* cb =
      (const NvtxExportTableCallbacks*)get_export_table(NVTX_ETID_CALLBACKS);
  NvtxFunctionTable table = 0;
  unsigned int size = 0;
  const char* path = getenv("OB_NVTX_LOG");
  if (!cb || !path || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE, &table, &size))
    return 0;
  if (size <= NVTX_CBID_CORE_RangePop) return 0;
  g_log = fopen(path, "w");
  if (!g_log) return 0;
  *table[NVTX_CBID_CORE_RangePushA] = (NvtxFunctionPointer)record_push;
  *table[NVTX_CBID_CORE_RangePop] = (NvtxFunctionPointer)record_pop;
  return 1;
}
