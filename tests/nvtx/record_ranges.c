/* An NVTX injection library for the tests: it records every range push and
 * pop of the process in the file named by DITSP_NVTX_LOG, one line each.
 * NVTX loads it when NVTX_INJECTION64_PATH names it, and calls
 * InitializeInjectionNvtx2, which installs the two handlers in NVTX's core
 * callback table. */
#include <stdio.h>
#include <stdlib.h>

#include <nvtx3/nvToolsExt.h>

static FILE* g_log;

static int NVTX_API record_push(const char* message) {
    if (g_log) {
        fprintf(g_log, "push %s\n", message ? message : "");
        fflush(g_log);
    }
    return 0;
}

static int NVTX_API record_pop(void) {
    if (g_log) {
        fprintf(g_log, "pop\n");
        fflush(g_log);
    }
    return 0;
}

int NVTX_API InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_export_table) {
    const char* path = getenv("DITSP_NVTX_LOG");
    g_log = fopen(path ? path : "/dev/null", "w");
    const NvtxExportTableCallbacks* cb = (const NvtxExportTableCallbacks*)get_export_table(NVTX_ETID_CALLBACKS);
    NvtxFunctionTable table = 0;
    unsigned int size = 0;
    if (!cb || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE, &table, &size)) return 0;
    if (size <= NVTX_CBID_CORE_RangePop) return 0;
    *table[NVTX_CBID_CORE_RangePushA] = (NvtxFunctionPointer)record_push;
    *table[NVTX_CBID_CORE_RangePop] = (NvtxFunctionPointer)record_pop;
    return 1;
}
