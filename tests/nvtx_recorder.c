/* A minimal NVTX tool for the tests: loaded by NVTX through
 * NVTX_INJECTION64_PATH, it records every range push and pop of the process,
 * one line each, to the file named by MOE_NVTX_LOG. Test infrastructure only. */
#include <stdio.h>
#include <stdlib.h>

#include <nvtx3/nvToolsExt.h>

static FILE* g_log;

static int record_push(const char* message)
{
    if (g_log) {
        fprintf(g_log, "push %s\n", message ? message : "");
        fflush(g_log);
    }
    return 0;
}

static int record_pop(void)
{
    if (g_log) {
        fprintf(g_log, "pop\n");
        fflush(g_log);
    }
    return 0;
}

/* Called by NVTX on the first NVTX call of the process. */
int InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_table)
{
    const NvtxExportTableCallbacks* cb = (const NvtxExportTableCallbacks*)get_table(NVTX_ETID_CALLBACKS);
    NvtxFunctionTable table = 0;
    unsigned int size = 0;
    if (!cb || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE, &table, &size) || size <= NVTX_CBID_CORE_RangePop)
        return 0;
    *table[NVTX_CBID_CORE_RangePushA] = (NvtxFunctionPointer)record_push;
    *table[NVTX_CBID_CORE_RangePop] = (NvtxFunctionPointer)record_pop;
    const char* path = getenv("MOE_NVTX_LOG");
    g_log = path ? fopen(path, "w") : 0;
    return 1;
}
