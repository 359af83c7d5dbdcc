/* A minimal NVTX tool for the tests: loaded through NVTX_INJECTION64_PATH, it
 * writes every domain creation and range push/pop of the process, one per line,
 * to the file named by KV_NVTX_LOG.  Built by tests/test_nvtx.py with the host
 * compiler; it uses only the public NVTX 3 headers of the CUDA toolkit. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

static FILE *log_file;

static const char *domain_name(nvtxDomainHandle_t d) { return d ? (const char *)d : "(default)"; }

static nvtxDomainHandle_t NVTX_API on_domain_create(const char *name) {
    fprintf(log_file, "domain %s\n", name);
    fflush(log_file);
    return (nvtxDomainHandle_t)strdup(name);
}

static int NVTX_API on_push(nvtxDomainHandle_t d, const nvtxEventAttributes_t *a) {
    const char *msg = a && a->messageType == NVTX_MESSAGE_TYPE_ASCII ? a->message.ascii : "?";
    fprintf(log_file, "push %s %s\n", domain_name(d), msg);
    fflush(log_file);
    return 0;
}

static int NVTX_API on_pop(nvtxDomainHandle_t d) {
    fprintf(log_file, "pop %s\n", domain_name(d));
    fflush(log_file);
    return 0;
}

int NVTX_API InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_table) {
    const char *path = getenv("KV_NVTX_LOG");
    const NvtxExportTableCallbacks *cb =
        (const NvtxExportTableCallbacks *)get_table(NVTX_ETID_CALLBACKS);
    NvtxFunctionTable t = 0;
    unsigned int last = 0;
    if (!path || !cb || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE2, &t, &last) ||
        last < NVTX_CBID_CORE2_DomainCreateA)
        return 0;
    log_file = fopen(path, "w");
    if (!log_file) return 0;
    *t[NVTX_CBID_CORE2_DomainCreateA] = (NvtxFunctionPointer)on_domain_create;
    *t[NVTX_CBID_CORE2_DomainRangePushEx] = (NvtxFunctionPointer)on_push;
    *t[NVTX_CBID_CORE2_DomainRangePop] = (NvtxFunctionPointer)on_pop;
    return 1;
}
