"""The bench's recorded-traffic lookup: a capture stays valid across comment
edits of the kernel sources and lapses when their code changes."""
import bench


def test_code_only_drops_comments_and_blank_lines():
    src = "int a = 1;  // one\n\n// a whole comment line\n  x += a;   \n"
    assert bench.code_only(src) == "int a = 1;\n  x += a;"


def test_comment_edit_keeps_the_hash_and_code_edit_changes_it():
    base = "__global__ void k() {\n    int a = 1;  // note\n}\n"
    comment_edit = "// header\n__global__ void k() {\n    int a = 1;  // another note\n\n}\n"
    code_edit = "__global__ void k() {\n    int a = 2;  // note\n}\n"
    assert bench.code_only(base) == bench.code_only(comment_edit)
    assert bench.code_only(base) != bench.code_only(code_edit)


def test_every_bench_kernel_name_maps_to_sources():
    for name in ("gemm_fprop", "quant_ffn_x", "block_quant_ffn_w", "ln_quant_ffn_x", "grouped_quant_moe_x"):
        assert len(bench.source_sha256(name)) == 64
