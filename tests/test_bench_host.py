"""Host-side helpers of bench.py (no GPU)."""
import bench


def test_code_only_drops_comments_and_whitespace():
    a = "int a = 1; // count\n/* block\n comment */ const char *s = \"//kept\";\n\n  char c = '/';"
    b = "int a = 1;\nconst char *s = \"//kept\"; char c = '/';"
    assert bench._code_only(a) == bench._code_only(b)
    assert '"//kept"' in bench._code_only(a)


def test_code_only_sees_code_changes():
    assert bench._code_only("x = a + b; // sum") != bench._code_only("x = a - b; // sum")
    assert bench._code_only('s = "a /* b */ c";') == 's = "a /* b */ c";'


def test_kernel_hashes_are_distinct_and_stable():
    hs = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    assert len(set(hs.values())) == len(hs)
    assert hs == {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
