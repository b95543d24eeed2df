/* A minimal NVTX tool for tests: loaded by the NVTX runtime from the path in
 * NVTX_INJECTION64_PATH, it appends one line per range push ("push <name>")
 * and pop ("pop") to the file named by MOE_NVTX_LOG.  Build:
 *   gcc -shared -fPIC -I<cuda>/include nvtx_injection.c -o libnvtx_injection.so */
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
    fputs("pop\n", g_log);
    fflush(g_log);
  }
  return 0;
}

int InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_export_table) {
  const NvtxExportTableCallbacks* cb =
      (const NvtxExportTableCallbacks*)get_export_table(NVTX_ETID_CALLBACKS);
  NvtxFunctionTable table = 0;
  unsigned int size = 0;
  const char* path = getenv("MOE_NVTX_LOG");
  if (!cb || !path || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE, &table, &size))
    return 0;
  if (size <= NVTX_CBID_CORE_RangePop) return 0;
  g_log = fopen(path, "w");
  if (!g_log) return 0;
  *table[NVTX_CBID_CORE_RangePushA] = (NvtxFunctionPointer)record_push;
  *table[NVTX_CBID_CORE_RangePop] = (NvtxFunctionPointer)record_pop;
  return 1;
}
