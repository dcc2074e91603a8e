"""W4A16 (bf16 activation x INT4 weight, group-128) linear layer for GB300."""
