"""B300-native paged GQA decode over a block-table KV cache, with GrowPage-style
page budgeting (scoring, top-k retention, compress-or-grow, compaction)."""
