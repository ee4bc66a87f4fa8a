/* Test infrastructure: an NVTX injection library that records the range pushes and pops of the
 * process that loads it. The NVTX code compiled into libwan.so loads the library named by
 * NVTX_INJECTION64_PATH at its first NVTX call and calls InitializeInjectionNvtx2, which here
 * points the core function table's RangePushA and RangePop entries at the two recorders below.
 * Each event becomes one line of the file named by WAN_NVTX_LOG: "push <name>" or "pop". */
#include <stdio.h>
#include <stdlib.h>

#include <nvtx3/nvToolsExt.h>

static FILE* g_log;

static int record_push(const char* name) {
  if (g_log) {
    fprintf(g_log, "push %s\n", name ? name : "(null)");
    fflush(g_log);
  }
  return 0;
}

static int record_pop(void) {
  if (g_log) {
    fputs("pop\n", g_log);
    fflush(g_log);
  }
  return 0;
}

int InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_export_table) {
  const char* path = getenv("WAN_NVTX_LOG");
  const NvtxExportTableCallbacks* cb =
      (const NvtxExportTableCallbacks*)get_export_table(NVTX_ETID_CALLBACKS);
  NvtxFunctionTable table = NULL;
  unsigned int size = 0;
  if (!path || !cb || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE, &table, &size) ||
      size <= NVTX_CBID_CORE_RangePop)
    return 0;
  g_log = fopen(path, "w");
  if (!g_log) return 0;
  *table[NVTX_CBID_CORE_RangePushA] = (NvtxFunctionPointer)record_push;
  *table[NVTX_CBID_CORE_RangePop] = (NvtxFunctionPointer)record_pop;
  return 1;
}
