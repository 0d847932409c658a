"""Host-side helpers of bench.py: the code-only source hash that ties an ncu
summary to the kernel source it measured."""
import bench


def test_code_only_drops_comments_and_layout_but_keeps_literals():
    src = 'int a;  // trailing\n/* block\n comment */ const char* s = "// kept /* kept */";\n\tchar c = \'"\';'
    assert bench.code_only(src) == 'int a; const char* s = "// kept /* kept */"; char c = \'"\';'


def test_source_hash_ignores_comment_edits_but_not_code_edits():
    base = {"a.cu": "__global__ void k(int* p) { p[0] = 1; }\n", "b.cuh": "#define X 3\n"}
    kinds = dict(bench.KERNEL_SOURCES)
    bench.KERNEL_SOURCES["_t"] = ["a.cu", "b.cuh"]
    try:
        h0 = bench.source_sha("_t", read=lambda rel: base[rel])
        commented = {"a.cu": "// a kernel\n__global__ void k(int* p) {\n  p[0] = 1;   /* one */\n}\n",
                     "b.cuh": "#define X 3  // three\n"}
        assert bench.source_sha("_t", read=lambda rel: commented[rel]) == h0
        changed = {"a.cu": "__global__ void k(int* p) { p[0] = 2; }\n", "b.cuh": "#define X 3\n"}
        assert bench.source_sha("_t", read=lambda rel: changed[rel]) != h0
        moved = {"a.cu": "__global__ void k(int* p) { p[0] = 1; }\n#define X 3\n", "b.cuh": ""}
        assert bench.source_sha("_t", read=lambda rel: moved[rel]) != h0   # file boundaries count
    finally:
        bench.KERNEL_SOURCES.clear()
        bench.KERNEL_SOURCES.update(kinds)
