"""Host logic of bench.py that needs no GPU: the source hash that decides
whether the committed ncu summary's DRAM bytes still describe the kernel, and
the prefill pass's FLOP count."""

import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_host", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_code_tokens_drop_comments_keep_literals():
    b = _bench()
    src = ('int a = 1;  // note "quoted"\n/* block\n comment */ const char* s = "// kept /* kept */";\n'
           "char q = '\"'; char e = '\\'';  int  b =\n 2;")
    assert b.code_tokens(src) == ('int a = 1; const char* s = "// kept /* kept */"; '
                                  "char q = '\"'; char e = '\\''; int b = 2;")


def test_kernel_hash_follows_code_not_comments(tmp_path):
    b = _bench()
    for f in b.KERNEL_SOURCES:
        os.makedirs(tmp_path / os.path.dirname(f), exist_ok=True)
        with open(os.path.join(ROOT, f)) as src, open(tmp_path / f, "w") as dst:
            dst.write(src.read())
    base = b.kernel_hash(str(tmp_path))
    assert base == b.kernel_hash()
    first = tmp_path / b.KERNEL_SOURCES[0]
    text = first.read_text()
    first.write_text("// a new comment line\n" + text.replace("\n", "  \n", 3))
    assert b.kernel_hash(str(tmp_path)) == base  # comments and spacing only
    first.write_text(text + "\nstatic int extra_symbol = 0;\n")
    assert b.kernel_hash(str(tmp_path)) != base  # code changed


def test_prefill_pairs_count_bottom_right_causal_keys():
    b = _bench()
    # brute force: new token j of a chunk of n ending a sequence of L tokens
    # sees keys 0 .. L - n + j
    for lens, qlens in (([5], [5]), ([9, 4], [3, 1]), ([40, 17, 33], [8, 17, 1])):
        brute = sum(L - n + j + 1 for L, n in zip(lens, qlens) for j in range(n))
        assert b.prefill_pairs(lens, qlens) == brute
    # the mixed step's two chunks: 917,760 + 1,966,336 pairs, 47.25 GFLOP at
    # 32 query heads x 4 x 128
    assert b.prefill_pairs([2048], [512]) == 917760
    assert b.prefill_pairs([4096], [512]) == 1966336
    assert b.prefill_pairs([2048, 4096], [512, 512]) * 32 * 4 * 128 == 47253028864
