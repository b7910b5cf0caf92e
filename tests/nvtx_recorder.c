/*
 * A minimal NVTX tool for the tracing test: loaded by the NVTX client code
 * compiled into libpagedattn (NVTX_INJECTION64_PATH names this library), it
 * subscribes to the domain calls of the NVTX core2 module and appends one line
 * per event to the file named by NVTX_RECORD_PATH:
 *
 *   create <domain>
 *   push <domain> <message>
 *   pop <domain>
 *
 * Only the public NVTX3 headers are used (the callback tables of
 * nvtxDetail/nvtxTypes.h).
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

typedef struct {
    char name[64];
} Domain;

static FILE *g_log;

static const char *domain_name(nvtxDomainHandle_t d) {
    return d ? ((const Domain *)d)->name : "(default)";
}

static nvtxDomainHandle_t on_domain_create(const char *name) {
    Domain *d = (Domain *)calloc(1, sizeof(Domain));
    if (!d) return NULL;
    strncpy(d->name, name ? name : "", sizeof(d->name) - 1);
    fprintf(g_log, "create %s\n", d->name);
    fflush(g_log);
    return (nvtxDomainHandle_t)d;
}

static int on_push(nvtxDomainHandle_t d, const nvtxEventAttributes_t *a) {
    const char *msg = (a && a->messageType == NVTX_MESSAGE_TYPE_ASCII && a->message.ascii)
                          ? a->message.ascii : "(none)";
    fprintf(g_log, "push %s %s\n", domain_name(d), msg);
    fflush(g_log);
    return 0;
}

static int on_pop(nvtxDomainHandle_t d) {
    fprintf(g_log, "pop %s\n", domain_name(d));
    fflush(g_log);
    return 0;
}

int InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_table) {
    const char *path = getenv("NVTX_RECORD_PATH");
    if (!path || !get_table) return 0;
    /* every NVTX client in the process (one per shared library that holds the
     * NVTX3 header code) loads this tool and calls this function once */
    if (!g_log) g_log = fopen(path, "a");
    if (!g_log) return 0;
    const NvtxExportTableCallbacks *cb =
        (const NvtxExportTableCallbacks *)get_table(NVTX_ETID_CALLBACKS);
    if (!cb || !cb->GetModuleFunctionTable) return 0;
    NvtxFunctionTable table = NULL;
    unsigned int size = 0;
    if (!cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE2, &table, &size) || !table) return 0;
    if (size < NVTX_CBID_CORE2_DomainCreateA) return 0;   /* size = highest valid index */
    *table[NVTX_CBID_CORE2_DomainCreateA] = (NvtxFunctionPointer)on_domain_create;
    *table[NVTX_CBID_CORE2_DomainRangePushEx] = (NvtxFunctionPointer)on_push;
    *table[NVTX_CBID_CORE2_DomainRangePop] = (NvtxFunctionPointer)on_pop;
    return 1;
}
