"""CPU tests of bench.py's host-side helpers (no GPU)."""
import bench


def test_strip_comments_keeps_code_and_literals():
    src = ('int a = 1; // one\n'
           '/* block\n   comment */ int b = 2;\n'
           'const char* s = "not // a comment";\n'
           "char c = '/';  /* x */\n"
           'asm("mma.sync /* inside a string */ ...");\n'
           '\n\n   \n'
           'int d = a / b;  // ratio\n')
    out = bench.strip_comments(src)
    assert out.splitlines() == ['int a = 1;', ' int b = 2;', 'const char* s = "not // a comment";',
                                "char c = '/';", 'asm("mma.sync /* inside a string */ ...");',
                                'int d = a / b;']


def test_kernel_hash_ignores_comment_edits(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    hdr = tmp_path / "k.cuh"
    src.write_text("// v1 comment\n__global__ void k() { int x = 1; }\n")
    hdr.write_text("static int y = 2;\n")
    monkeypatch.setattr(bench, "KERNEL_SRC", str(src))
    monkeypatch.setattr(bench, "KERNEL_HDR", str(hdr))
    h1 = bench.kernel_src_sha()
    src.write_text("// reworded comment\n\n__global__ void k() { int x = 1; }  /* note */\n")
    assert bench.kernel_src_sha() == h1
    src.write_text("__global__ void k() { int x = 2; }\n")
    assert bench.kernel_src_sha() != h1

