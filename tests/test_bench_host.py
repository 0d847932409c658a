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


# --- algorithmic work behind every roofline figure -----------------------------
from types import SimpleNamespace


def _shape(**kw):
    n_valid = kw.pop("n_valid", 0)
    return SimpleNamespace(n_valid=lambda: n_valid, **kw)


def test_decode_bytes_of_the_default_workload():
    # 4 slices x 16,384 listed rows, 8 KV heads, D 128, bf16: K + V = 512 B per (row, head)
    p = _shape(n_valid=4 * 16384, Hkv=8, D=128)
    assert bench.decode_bytes(p) == 268_435_456


def test_decode_bytes_of_the_small_and_sparse_workloads():
    assert bench.decode_bytes(_shape(n_valid=2 * 1000, Hkv=2, D=128)) == 2_048_000
    assert bench.decode_bytes(_shape(n_valid=2048, Hkv=2, D=256)) == 4_194_304


def test_quantised_decode_bytes_count_codes_and_two_scales():
    p = _shape(n_valid=1000, Hkv=8, D=128)
    assert bench.decode_bytes(p, "int8") == 1000 * 8 * (256 + 4)
    assert bench.decode_bytes(p, "fp8") == 1000 * 8 * (256 + 4)
    assert bench.decode_bytes(p, "int4") == 1000 * 8 * (128 + 4)


def test_prefill_flops_closed_form_of_the_prefill_workload():
    # 4 x 2,048 causal queries (bottom-right) over 99,936-row lists, 32 query heads, D 128:
    # visible pairs per (slice, head) = 2048 * (99936 - 2048) + 2048 * 2049 / 2
    p = SimpleNamespace(L=99936, Nq=2048, D=128, Hq=32, S=4)
    pairs = 2048 * (99936 - 2048) + 2048 * 2049 // 2
    assert pairs == 202_572_800                      # = 2048 * 97,889 + 2047 * 2048 / 2
    assert bench.prefill_flops(p) == 4 * 128 * 32 * 4 * pairs == 13_275_811_020_800


def test_prefill_flops_brute_force_on_a_tiny_case():
    p = SimpleNamespace(L=7, Nq=3, D=2, Hq=1, S=1)
    visible = sum(1 for i in range(3) for j in range(7) if j <= 7 - 3 + i)
    assert bench.prefill_flops(p) == 4 * 2 * visible


def test_append_bytes_count_input_codes_scale_and_index():
    assert bench.append_bytes(8192, 8, 128) == 8192 * (8 * (256 + 128 + 2) + 4) == 25_329_664
