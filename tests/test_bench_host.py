"""Host logic of bench.py that needs no GPU: the GEMM source hash that keys
the recorded DRAM-traffic lines ignores comments and blank lines, and
nothing else."""

import bench


def test_code_only_drops_comments_and_blank_lines():
    src = ('int a = 1;  // a comment\n'
           '/* a block\n   comment */ char s[] = "x // not a comment /* nor this */";\n'
           "char q = '\"'; char e = '\\\\';\n"
           '\n'
           '   \n'
           'int b = 2;   \n')
    assert bench.code_only(src) == (
        'int a = 1;\n'
        ' char s[] = "x // not a comment /* nor this */";\n'
        "char q = '\"'; char e = '\\\\';\n"
        'int b = 2;')


def test_comment_edits_keep_the_hash_and_code_edits_change_it():
    a = 'int f(int x) {\n    return x + 1;  // the successor\n}\n'
    b = '// f: the successor\nint f(int x) {\n\n    return x + 1;\n}\n'
    c = 'int f(int x) {\n    return x + 2;  // the successor\n}\n'
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)

